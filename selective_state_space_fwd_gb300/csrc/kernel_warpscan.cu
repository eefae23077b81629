// kernel_warpscan.cu -- the WARPSCAN tier of libssmscan: the hierarchical
// parallel scan of [P1] s3.1 mapped onto a warp.
//
// One warp owns one (b, d) channel.  The sequence is cut into windows of
// W = 32 * K steps; lane l owns the K consecutive steps [l K, l K + K) of a
// window ([P1] s3.1 first level: a thread-serial run in registers).  For each
// pair of states the warp then
//   1. folds its K steps serially into one affine pair (a_prod, b_sum) with the
//      combine (a1,b1) o (a2,b2) = (a1 a2, a2 b1 + b2) ([P1] s2.1, [P2] s2.2),
//      keeping every step's (a, b) in registers;
//   2. runs a 5-round Hillis-Steele inclusive scan of the lanes' pairs with
//      __shfl_up_sync, updating b before a ([P1] s2.2, s4.2: the b update reads
//      the old a), so lane l holds the composition of lanes 0..l;
//   3. applies the window's incoming state (the serial carry between windows,
//      [P1] s3.1 third level, [P2] s2.4) to get the state before its run, and
//      replays its K steps from registers: h = a h + b, y += C h ([P1] s3.3:
//      the state never leaves registers).
// After all states the lane adds D x, applies the silu(z) gate and writes y.
// Padded steps (t >= valid_len, or past L) are folded into the identity
// (a = 1, b = 0) by zeroing delta and x ([P1] s2.3, s5.3).
//
// Block: 4 warps = 4 consecutive channels of one batch row, sharing the
// window's B and C rows in shared memory.  x, delta, z are staged transposed
// per channel so that a lane's K steps are contiguous.  Shared-memory layouts
// are XOR-swizzled so the lane-strided reads are conflict-free.
#include "common.cuh"
#include "tiers.h"

namespace ssm {
namespace {

typedef unsigned long long u64;

__device__ __forceinline__ u64 pk2(float lo, float hi) {
  u64 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 upk2(u64 v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ u64 mul2(u64 a, u64 b) {
  u64 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ u64 fma2(u64 a, u64 b, u64 c) {
  u64 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ u64 shfl_up2(u64 v, int delta) {
  const float2 f = upk2(v);
  return pk2(__shfl_up_sync(0xffffffffu, f.x, delta), __shfl_up_sync(0xffffffffu, f.y, delta));
}
__device__ __forceinline__ u64 shfl_idx2(u64 v, int src) {
  const float2 f = upk2(v);
  return pk2(__shfl_sync(0xffffffffu, f.x, src), __shfl_sync(0xffffffffu, f.y, src));
}

// Asynchronous global -> shared copies of 4 or 8 bytes (cp.async); when `pred`
// is false nothing is read and the destination is zero-filled.
__device__ __forceinline__ void cp_async4(float* dst, const float* src, bool pred) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(pred ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async8(float* dst, const float* src, bool pred) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(pred ? 8 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

constexpr int kWarps = 4;  // channels per block
constexpr int kQ = 2;      // state pairs interleaved per pass

// Position of step r of a per-channel row in shared memory.  Lane l = r / K
// owns K consecutive steps; with K = 8 its two float4 halves are stored in an
// order set by bit 2 of l, so a quarter-warp of 16-byte loads covers all 32
// banks.  With K = 4 the natural order is already conflict-free.
template <int K>
__device__ __forceinline__ int act_pos(int r) {
  if (K == 4) return r;
  const int l = r >> 3, j = r & 7;
  const int half = (j >> 2) ^ ((l >> 2) & 1);
  return l * 8 + half * 4 + (j & 3);
}

// Swizzled column of state n in a B / C row read by lane l: an XOR with an even
// value keeps (n, n+1) pairs together and 8-byte aligned, and spreads the
// lane-strided rows over the banks.
template <int N>
__device__ __forceinline__ int bc_col(int n, int l) {
  return n ^ ((l & (N / 2 - 1)) << 1);
}

template <int N>
struct WShape {
  static constexpr int K = N >= 64 ? 4 : 8;  // steps per lane run
  static constexpr int W = 32 * K;           // steps per window
};

template <int N, typename T>
struct WCfg {
  static constexpr int K = WShape<N>::K, W = WShape<N>::W;
  static constexpr int ACT = kWarps * W;  // floats of one transposed x / delta / z / y tile
  static constexpr int BC = W * N;        // floats of one B / C tile
  static constexpr int SMEM = (4 * ACT + 2 * BC + kWarps * N) * 4;
};

// Load this lane's K consecutive entries of a transposed per-channel tile.
template <int K>
__device__ __forceinline__ void load_run(const float* tile, int lane, float (&v)[K]) {
  const float4* t4 = reinterpret_cast<const float4*>(tile);
  if (K == 4) {
    const float4 a = t4[lane];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  } else {
    const int sw = (lane >> 2) & 1;
    const float4 a = t4[lane * 2 + sw], c = t4[lane * 2 + (sw ^ 1)];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
  }
}

// ASYNC: fp32 inputs with 8-byte aligned B and C, staged with cp.async.
template <int N, typename T, bool GATE, bool ASYNC>
__global__ void __launch_bounds__(kWarps * 32) warpscan_kernel(const ScanParams p) {
  using C = WCfg<N, T>;
  constexpr int K = C::K, W = C::W;
  extern __shared__ __align__(16) float sm[];
  float* xs = sm;                    // [warp][act_pos(r)]
  float* ds = xs + C::ACT;
  float* zs = ds + C::ACT;
  float* ys = zs + C::ACT;
  float* bs = ys + C::ACT;           // [r][bc_col(n, r / K)]
  float* cs = bs + C::BC;
  float* carry = cs + C::BC;         // [warp][N]: state entering the window

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n_cg = (p.dim + kWarps - 1) / kWarps;
  const int64_t b = blockIdx.x / n_cg;
  const int64_t d0 = (blockIdx.x % n_cg) * kWarps;
  const int64_t d = d0 + warp;
  const bool d_ok = d < p.dim;
  const int64_t L = p.seqlen;
  const int64_t lv = valid_steps(p, b);
  const float dskip = (d_ok && p.D) ? __ldg(p.D + d) : 0.f;
  const float dbias = d_ok ? delta_bias(p.dt_bias, d) : 0.f;
  const bool want_states = p.states != nullptr;
  const int row0 = lane * K;

  for (int i = threadIdx.x; i < kWarps * N; i += blockDim.x) {  // h_0 = 0 unless given
    const int64_t dc = d0 + i / N;
    carry[i] = (p.h0 && dc < p.dim) ? __ldg(p.h0 + (b * p.dim + dc) * N + i % N) : 0.f;
  }

  for (int64_t t0 = 0; t0 < L; t0 += W) {
    const int nw = static_cast<int>(L - t0 < W ? L - t0 : W);  // steps of this window
    const int64_t rem = lv - t0;
    const int nv = static_cast<int>(rem <= 0 ? 0 : (rem < nw ? rem : nw));  // valid steps
    __syncthreads();  // the previous window is fully consumed
    if (nv > 0) {
      // Stage the window: x, delta (, z) transposed per channel, B and C rows
      // (steps past the valid length are zero-filled: identity steps).
      if constexpr (ASYNC) {
        const float* gx = static_cast<const float*>(p.x);
        const float* gd = static_cast<const float*>(p.delta);
        const float* gz = static_cast<const float*>(p.z);
        const float* gb = static_cast<const float*>(p.B);
        const float* gc = static_cast<const float*>(p.C);
        for (int r = threadIdx.x; r < W; r += blockDim.x) {
          const bool in = r < nv;
          const int pos = act_pos<K>(r);
          const int64_t e = in ? (b * L + t0 + r) * p.dim + d0 : 0;
#pragma unroll
          for (int c = 0; c < kWarps; ++c) {
            const bool ok = in && d0 + c < p.dim;
            cp_async4(xs + c * W + pos, gx + (ok ? e + c : 0), ok);
            cp_async4(ds + c * W + pos, gd + (ok ? e + c : 0), ok);
            if (GATE) cp_async4(zs + c * W + pos, gz + (ok ? e + c : 0), ok);
          }
        }
        for (int i = threadIdx.x; i < W * N / 2; i += blockDim.x) {  // state pairs
          const int r = (2 * i) / N, n = (2 * i) % N;
          const bool in = r < nv;
          const int64_t e = in ? (b * L + t0 + r) * N + n : 0;
          const int col = bc_col<N>(n, r / K);
          cp_async8(bs + r * N + col, gb + e, in);
          cp_async8(cs + r * N + col, gc + e, in);
        }
        cp_async_wait_all();
      } else {
        for (int r = threadIdx.x; r < W; r += blockDim.x) {
          const bool in = r < nv;
          const int pos = act_pos<K>(r);
          const int64_t e = (b * L + t0 + r) * p.dim + d0;
#pragma unroll
          for (int c = 0; c < kWarps; ++c) {
            const bool ok = in && d0 + c < p.dim;
            xs[c * W + pos] = ok ? IO<T>::load(p.x, e + c) : 0.f;
            ds[c * W + pos] = ok ? IO<T>::load(p.delta, e + c) : 0.f;
            if (GATE) zs[c * W + pos] = ok ? IO<T>::load(p.z, e + c) : 0.f;
          }
        }
        for (int i = threadIdx.x; i < W * N / 2; i += blockDim.x) {  // state pairs
          const int r = (2 * i) / N, n = (2 * i) % N;
          const bool in = r < nv;
          const int64_t e = (b * L + t0 + r) * N + n;
          const int col = bc_col<N>(n, r / K);
          float2 bv = make_float2(0.f, 0.f), cv = make_float2(0.f, 0.f);
          if (in) {
            bv = make_float2(IO<T>::load(p.B, e), IO<T>::load(p.B, e + 1));
            cv = make_float2(IO<T>::load(p.C, e), IO<T>::load(p.C, e + 1));
          }
          *reinterpret_cast<float2*>(bs + r * N + col) = bv;
          *reinterpret_cast<float2*>(cs + r * N + col) = cv;
        }
      }
      __syncthreads();

      // This lane's K steps.
      float dt[K], xv[K];
      load_run<K>(ds + warp * W, lane, dt);
      load_run<K>(xs + warp * W, lane, xv);
      if (has_delta_prep(p)) {  // bias, softplus, clipping; padded steps stay 0
#pragma unroll
        for (int j = 0; j < K; ++j)
          if (row0 + j < nv) dt[j] = prep_delta(dt[j], dbias, p);
      }
      u64 dd[K], uu[K], y2[K];
#pragma unroll
      for (int j = 0; j < K; ++j) {
        const float u = dt[j] * xv[j];
        dd[j] = pk2(dt[j], dt[j]);
        uu[j] = pk2(u, u);
        y2[j] = pk2(0.f, 0.f);
      }
      // first chunk-end step at or after this lane's run ([P1] s3.4)
      int64_t ce0 = INT64_MAX;
      if (want_states) {
        const int64_t ts = t0 + row0;
        ce0 = (ts / p.chunk_len + 1) * p.chunk_len - 1;
        if (ce0 > L - 1) ce0 = L - 1;
      }
      const bool run_has_ce = ce0 < t0 + row0 + K;

      // kQ state pairs per pass: their folds, scans and replays are independent,
      // so their shuffle and MUFU latencies overlap.
      for (int n0 = 0; n0 < N; n0 += 2 * kQ) {
        int col[kQ];
        u64 a2[kQ];
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
          const int n = n0 + 2 * q;
          col[q] = bc_col<N>(n, lane);
          float alo = 0.f, ahi = 0.f;
          if (d_ok) {
            alo = __ldg(p.A + d * N + n) * kLog2e;
            ahi = __ldg(p.A + d * N + n + 1) * kLog2e;
          }
          a2[q] = pk2(alo, ahi);
        }
        // 1. thread-serial fold of the lane's K steps, keeping each (a, b)
        u64 av[kQ][K], bv[kQ][K], A[kQ], Bsum[kQ];
#pragma unroll
        for (int j = 0; j < K; ++j) {
#pragma unroll
          for (int q = 0; q < kQ; ++q) {
            const u64 bq = *reinterpret_cast<const u64*>(bs + (row0 + j) * N + col[q]);
            const float2 arg = upk2(mul2(a2[q], dd[j]));
            av[q][j] = pk2(ex2(arg.x), ex2(arg.y));  // Abar = exp(delta A)
            bv[q][j] = mul2(bq, uu[j]);               // delta B x
            if (j == 0) {
              A[q] = av[q][0];
              Bsum[q] = bv[q][0];
            } else {  // (A, Bsum) o (a_j, b_j)
              Bsum[q] = fma2(av[q][j], Bsum[q], bv[q][j]);
              A[q] = mul2(A[q], av[q][j]);
            }
          }
        }
        // 2. 5-round Hillis-Steele inclusive scan across the warp, b before a
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
          for (int q = 0; q < kQ; ++q) {
            const u64 Aup = shfl_up2(A[q], off), Bup = shfl_up2(Bsum[q], off);
            if (lane >= off) {
              Bsum[q] = fma2(A[q], Bup, Bsum[q]);  // b = a_self * b_prev + b_self (old a)
              A[q] = mul2(A[q], Aup);
            }
          }
        }
        // 3. window carry: the state before this lane's run, then the replay
        u64 h[kQ], hlast[kQ];
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
          const int n = n0 + 2 * q;
          const u64 hin = pk2(carry[warp * N + n], carry[warp * N + n + 1]);
          const u64 hend = fma2(A[q], hin, Bsum[q]);  // state after this lane's run
          h[q] = shfl_up2(hend, 1);
          if (lane == 0) h[q] = hin;
          hlast[q] = shfl_idx2(hend, 31);  // state entering the next window
        }
        int64_t ce = ce0;
#pragma unroll
        for (int j = 0; j < K; ++j) {
#pragma unroll
          for (int q = 0; q < kQ; ++q) {
            h[q] = fma2(av[q][j], h[q], bv[q][j]);
            const u64 cq = *reinterpret_cast<const u64*>(cs + (row0 + j) * N + col[q]);
            y2[j] = fma2(cq, h[q], y2[j]);
          }
          if (run_has_ce && t0 + row0 + j == ce) {  // [P1] s3.4 chunk boundary state
            if (d_ok) {
#pragma unroll
              for (int q = 0; q < kQ; ++q) {
                float* sp = p.states +
                            ((b * p.n_chunks + ce / p.chunk_len) * p.dim + d) * N + n0 + 2 * q;
                *reinterpret_cast<float2*>(sp) = upk2(h[q]);
              }
            }
            ce = ce + p.chunk_len > L - 1 ? (ce == L - 1 ? INT64_MAX : L - 1) : ce + p.chunk_len;
          }
        }
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int q = 0; q < kQ; ++q)
            *reinterpret_cast<float2*>(carry + warp * N + n0 + 2 * q) = upk2(hlast[q]);
        }
        __syncwarp();
      }
      // epilogue: y = (sum_n C h + D x) * silu(z); exact 0 at identity steps
      float zv[K];
      if (GATE) load_run<K>(zs + warp * W, lane, zv);
#pragma unroll
      for (int j = 0; j < K; ++j) {
        const float2 ya = upk2(y2[j]);
        float yv = fmaf(dskip, xv[j], ya.x + ya.y);
        if (GATE) yv *= silu(zv[j]);
        if (row0 + j >= nv) yv = 0.f;
        ys[warp * W + act_pos<K>(row0 + j)] = yv;
      }
      __syncthreads();
      for (int r = threadIdx.x; r < nw; r += blockDim.x) {  // y rows, channels contiguous
        const int64_t e = (b * L + t0 + r) * p.dim + d0;
        const int pos = act_pos<K>(r);
#pragma unroll
        for (int c = 0; c < kWarps; ++c)
          if (d0 + c < p.dim) IO<T>::store(p.y, e + c, ys[c * W + pos]);
      }
    } else {
      // Whole window past the valid length: y = 0, chunk states frozen.
      for (int r = threadIdx.x; r < nw; r += blockDim.x) {
        const int64_t e = (b * L + t0 + r) * p.dim + d0;
#pragma unroll
        for (int c = 0; c < kWarps; ++c)
          if (d0 + c < p.dim) IO<T>::store(p.y, e + c, 0.f);
      }
      if (want_states && d_ok) {
        int64_t ce = (t0 / p.chunk_len + 1) * p.chunk_len - 1;
        if (ce > L - 1) ce = L - 1;
        while (ce < t0 + nw) {
          float* sp = p.states + ((b * p.n_chunks + ce / p.chunk_len) * p.dim + d) * N;
          for (int n = lane; n < N; n += 32) sp[n] = carry[warp * N + n];
          if (ce == L - 1) break;
          ce = ce + p.chunk_len > L - 1 ? L - 1 : ce + p.chunk_len;
        }
      }
    }
  }
  if (p.h_final) {  // state after the last step
    __syncthreads();
    for (int i = threadIdx.x; i < kWarps * N; i += blockDim.x) {
      const int64_t dc = d0 + i / N;
      if (dc < p.dim) p.h_final[(b * p.dim + dc) * N + i % N] = carry[i];
    }
  }
}

template <int N, typename T>
cudaError_t launch_nt(const ScanParams& p, cudaStream_t s) {
  using C = WCfg<N, T>;
  static bool attr_done[4] = {false, false, false, false};
  const int64_t grid = (p.dim + kWarps - 1) / kWarps * p.batch;
  constexpr bool kF32 = sizeof(T) == 4;
  const bool async = kF32 && (reinterpret_cast<uintptr_t>(p.B) % 8 == 0) &&
                     (reinterpret_cast<uintptr_t>(p.C) % 8 == 0);
  const int gi = (p.z ? 1 : 0) + (async ? 2 : 0);
  auto kern = async ? (p.z ? warpscan_kernel<N, T, true, kF32> : warpscan_kernel<N, T, false, kF32>)
                    : (p.z ? warpscan_kernel<N, T, true, false> : warpscan_kernel<N, T, false, false>);
  if (!attr_done[gi]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_done[gi] = true;
  }
  kern<<<static_cast<unsigned>(grid), kWarps * 32, C::SMEM, s>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const ScanParams& p, cudaStream_t s) {
  switch (p.dstate) {
    case 8: return launch_nt<8, T>(p, s);
    case 16: return launch_nt<16, T>(p, s);
    case 32: return launch_nt<32, T>(p, s);
    case 64: return launch_nt<64, T>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool warpscan_eligible(const ScanParams& p) {
  if (p.dstate != 8 && p.dstate != 16 && p.dstate != 32 && p.dstate != 64) return false;
  const int64_t grid = (p.dim + kWarps - 1) / kWarps * p.batch;
  return grid <= INT32_MAX;
}

int64_t warpscan_grid(const ScanParams& p) { return (p.dim + kWarps - 1) / kWarps * p.batch; }

cudaError_t launch_warpscan(const ScanParams& p, bool bf16, cudaStream_t s) {
  return bf16 ? launch_t<__nv_bfloat16>(p, s) : launch_t<float>(p, s);
}

}  // namespace ssm
