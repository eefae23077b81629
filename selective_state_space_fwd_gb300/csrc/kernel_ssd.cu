// kernel_ssd.cu -- the SSD form of the scan (one decay per head) on the
// tensor cores ([P2] s5.1-s5.2: the recurrence expanded into a semiseparable
// matrix product; blocks of steps done as matrix products, the state carried
// from block to block by the recurrence itself).
//
// Per head h with decay a_t = exp(delta_t A_h) and a block of Q = 128 steps,
// write cs_t = sum_{r<=t} delta_r A_h (in log2 units) inside the block and
// S for the state entering it ([N x P]: state n, channel p of the head):
//   G'[t,s] = C_t . (delta_s B_s)                          (tensor cores, K = N)
//   Ym[t,s] = G'[t,s] 2^(cs_t - cs_s) for s <= t, else 0   (registers)
//   Yd      = Ym x                                         (tensor cores, K = Q)
//   Yo      = C S                                          (tensor cores, K = N)
//   y_t     = (Yd_t + 2^cs_t Yo_t + D x_t) silu(z_t)
//   S      <- 2^cs_end S + (delta B)^T (2^(cs_end - cs_s) x_s)   (tensor cores, K = Q)
// which is the recurrence regrouped: the output of step t is the inputs of
// the block weighted by the decay between their step and t, plus the state
// entering the block decayed to t.  Operands are bf16 in shared memory in
// the non-swizzled core-matrix layout (umma.cuh), products accumulate in
// fp32 in tensor memory, and the state stays fp32 in registers between
// blocks (rounded to bf16 only as an operand of Yo).
//
// One CTA of 128 threads per (batch row, head), blocks in order.  Thread i is
// step i of the block when staging and in the epilogue (TMEM lane i holds row
// i of G', Yd and Yo) and state row i for the state update (lane i of dS).
// Shared memory is about 113 KB, so two CTAs share an SM and one CTA's
// staging and epilogue overlap the other's matrix products.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ssd.h"
#include "umma.cuh"

namespace ssm {
namespace {

constexpr int Q = kSsdChunk, P = kSsdHeadDim, N = kSsdState;
constexpr int kThreads = 128;
constexpr unsigned kSsdWaitLimit = 1u << 24;  // try_wait polls before a wait gives up
constexpr unsigned kErrSsdWait = 2u;
static_assert(N == Q, "the C / B tile and the masked-G tile share one layout");

// Tiles (byte offsets in dynamic shared memory).  A K-major [rows x K] tile
// puts core matrix (r8, k8) at r8 * (K / 8) * 128 + k8 * 128; an MN-major
// tile of MN extent E puts core matrix (mn8, k8) at k8 * (E / 8) * 128 + mn8 * 128.
constexpr uint32_t kTileC = 0;                    // C rows, K-major [t x n]
constexpr uint32_t kTileB = kTileC + Q * N * 2;   // delta-scaled B rows, K-major [s x n]; then Ym [t x s]
constexpr uint32_t kTileX = kTileB + Q * N * 2;   // x, MN-major [p x s]
constexpr uint32_t kTileXw = kTileX + Q * P * 2;  // x decayed to the block end, MN-major [p x s]
constexpr uint32_t kTileS = kTileXw + Q * P * 2;  // state entering the block, MN-major [p x n]
constexpr uint32_t kCs = kTileS + N * P * 2;      // cs per step of the block, fp32 [Q]
constexpr uint32_t kDs = kCs + Q * 4;             // D of the head's channels, fp32 [P]
constexpr uint32_t kWarpTot = kDs + P * 4;        // per-warp totals of the scan of cs
constexpr uint32_t kBar = kWarpTot + 16;          // mbarrier
constexpr uint32_t kSlot = kBar + 8;              // TMEM base address
constexpr uint32_t kSmemBytes = kSlot + 8;
constexpr uint32_t kRowK = (N / 8) * 128;  // core-matrix row stride of the K-major tiles (2048)
constexpr uint32_t kRowX = (P / 8) * 128;  // K-direction stride of the MN-major tiles (1024)

// TMEM columns (fp32): G' [0,128) then Yd [0,64); Yo [128,192); dS [192,256).
constexpr uint32_t kColG = 0, kColYd = 0, kColYo = 128, kColDS = 192, kTmemCols = 256;

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ uint4 pack8(const float* f) {
  return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
}
__device__ __forceinline__ void sts128(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ uint4 ldg128(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

template <bool GATE>
__global__ void __launch_bounds__(kThreads, 2) ssd_kernel(const SsdParams p) {
  extern __shared__ __align__(1024) unsigned char sm[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t H = p.nheads, L = p.seqlen, Dm = p.nheads * P;
  const int64_t b = blockIdx.x / H, h = blockIdx.x % H;
  const uint32_t s0 = umma::smem_u32(sm);
  const uint32_t bar = s0 + kBar;
  float* sCs = reinterpret_cast<float*>(sm + kCs);
  float* sD = reinterpret_cast<float*>(sm + kDs);
  float* sWt = reinterpret_cast<float*>(sm + kWarpTot);
  const auto* xg = static_cast<const __nv_bfloat16*>(p.x);
  const auto* zg = static_cast<const __nv_bfloat16*>(p.z);
  const auto* Bg = static_cast<const __nv_bfloat16*>(p.B);
  const auto* Cg = static_cast<const __nv_bfloat16*>(p.C);
  auto* yg = static_cast<__nv_bfloat16*>(p.y);

  if (warp == 0) umma::tmem_alloc(s0 + kSlot, kTmemCols);
  if (tid == 0) umma::mbar_init(bar, 1);
  if (tid < P) sD[tid] = p.D ? __ldg(p.D + h * P + tid) : 0.f;
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tm = *reinterpret_cast<volatile uint32_t*>(sm + kSlot);
  const uint32_t tl = tm + (static_cast<uint32_t>(warp * 32) << 16);  // this warp's TMEM lanes

  int64_t Lv = L;
  if (p.valid_len) {
    Lv = p.valid_len[b];
    Lv = Lv < 0 ? 0 : (Lv > L ? L : Lv);
  }
  const float al = __ldg(p.A + h) * kLog2e;  // A_h in log2 units

  // S[n][p] for this thread's state row n = tid
  float S[P];
#pragma unroll
  for (int j = 0; j < P; ++j) S[j] = p.h0 ? p.h0[((b * Dm + h * P + j) * N) + tid] : 0.f;

  uint32_t phase = 0;
  bool bad = false;
  for (int64_t t0 = 0; t0 < L; t0 += Q) {
    const int64_t t = t0 + tid;
    const bool in = t < Lv;  // a valid step (Lv <= L)
    const int64_t row = b * L + t;
    if (t0 >= Lv) {  // the whole block is past valid_len: output 0, state frozen
      if (t < L) {
#pragma unroll
        for (int c = 0; c < P / 8; ++c)
          *reinterpret_cast<uint4*>(yg + row * Dm + h * P + c * 8) = make_uint4(0, 0, 0, 0);
      }
      continue;
    }
    // step size and the inclusive scan of delta A over the block
    const float dt = in ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.delta)[row * H + h]) : 0.f;
    float cs = dt * al;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float v = __shfl_up_sync(0xFFFFFFFFu, cs, o);
      if (lane >= o) cs += v;
    }
    if (lane == 31) sWt[warp] = cs;
    __syncthreads();
    float pre = 0.f, tot = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
      const float v = sWt[w];
      pre += w < warp ? v : 0.f;
      tot += v;
    }
    cs += pre;
    sCs[tid] = cs;
    const float wend = ex2(tot - cs);  // decay from step t to the end of the block

    // stage this step's rows (zero rows past valid_len, so that nothing there
    // reaches a product)
    const uint32_t rk = (tid >> 3) * kRowK + (tid & 7) * 16;  // row tid of a K-major tile
    const uint32_t rx = (tid >> 3) * kRowX + (tid & 7) * 16;  // K-row tid of an MN-major tile
#pragma unroll
    for (int c = 0; c < N / 8; ++c) {
      const uint4 v = in ? ldg128(Cg + row * N + c * 8) : make_uint4(0, 0, 0, 0);
      sts128(s0 + kTileC + rk + c * 128, v);
    }
#pragma unroll
    for (int c = 0; c < N / 8; ++c) {
      const uint4 v = in ? ldg128(Bg + row * N + c * 8) : make_uint4(0, 0, 0, 0);
      float f[8];
      unpack8(v, f);
#pragma unroll
      for (int j = 0; j < 8; ++j) f[j] *= dt;
      sts128(s0 + kTileB + rk + c * 128, pack8(f));
    }
    uint4 zr[GATE ? P / 8 : 1];
#pragma unroll
    for (int c = 0; c < P / 8; ++c) {
      const uint4 v = in ? ldg128(xg + row * Dm + h * P + c * 8) : make_uint4(0, 0, 0, 0);
      sts128(s0 + kTileX + rx + c * 128, v);
      float f[8];
      unpack8(v, f);
#pragma unroll
      for (int j = 0; j < 8; ++j) f[j] *= wend;
      sts128(s0 + kTileXw + rx + c * 128, pack8(f));
      if (GATE) zr[c] = in ? ldg128(zg + row * Dm + h * P + c * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int c = 0; c < P / 8; ++c) sts128(s0 + kTileS + rx + c * 128, pack8(S + c * 8));
    umma::fence_smem_to_async();
    umma::fence_before_sync();
    __syncthreads();

    if (tid == 0) {
      umma::fence_after_sync();
      constexpr uint32_t idG = umma::idesc_bf16(128, Q, false, false);
      constexpr uint32_t idO = umma::idesc_bf16(128, P, false, true);
      constexpr uint32_t idS = umma::idesc_bf16(128, P, true, true);
#pragma unroll
      for (int k = 0; k < N / 16; ++k)  // G' = C (delta B)^T
        umma::mma_bf16(tm + kColG, umma::smem_desc(s0 + kTileC + k * 256, 128, kRowK),
                       umma::smem_desc(s0 + kTileB + k * 256, 128, kRowK), idG, k > 0);
#pragma unroll
      for (int k = 0; k < N / 16; ++k)  // Yo = C S
        umma::mma_bf16(tm + kColYo, umma::smem_desc(s0 + kTileC + k * 256, 128, kRowK),
                       umma::smem_desc(s0 + kTileS + k * 2 * kRowX, kRowX, 128), idO, k > 0);
#pragma unroll
      for (int k = 0; k < Q / 16; ++k)  // dS = (delta B)^T (x decayed to the block end)
        umma::mma_bf16(tm + kColDS, umma::smem_desc(s0 + kTileB + k * 2 * kRowK, kRowK, 128),
                       umma::smem_desc(s0 + kTileXw + k * 2 * kRowX, kRowX, 128), idS, k > 0);
      umma::mma_commit(bar);
    }
    __syncwarp();
    if (!umma::mbar_wait(bar, phase, kSsdWaitLimit)) bad = true;
    phase ^= 1;
    if (__syncthreads_or(bad)) { bad = true; break; }
    umma::fence_after_sync();

    // Ym row t = tid into the B tile (its products are done)
#pragma unroll
    for (int sb = 0; sb < Q / 32; ++sb) {
      uint4 o[4];
      if (sb <= warp) {  // warp-uniform: columns past the warp's last row are all masked
        float g[32];
        umma::tmem_ld32(tl + kColG + sb * 32, g);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int s = sb * 32 + j;
          g[j] = s <= tid ? g[j] * ex2(cs - sCs[s]) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) o[q] = pack8(g + q * 8);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) o[q] = make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) sts128(s0 + kTileB + rk + (sb * 4 + q) * 128, o[q]);
    }
    umma::fence_smem_to_async();
    umma::fence_before_sync();
    __syncthreads();

    if (tid == 0) {
      umma::fence_after_sync();
      constexpr uint32_t idY = umma::idesc_bf16(128, P, false, true);
#pragma unroll
      for (int k = 0; k < Q / 16; ++k)  // Yd = Ym x
        umma::mma_bf16(tm + kColYd, umma::smem_desc(s0 + kTileB + k * 256, 128, kRowK),
                       umma::smem_desc(s0 + kTileX + k * 2 * kRowX, kRowX, 128), idY, k > 0);
      umma::mma_commit(bar);
    }
    __syncwarp();
    if (!umma::mbar_wait(bar, phase, kSsdWaitLimit)) bad = true;
    phase ^= 1;
    if (__syncthreads_or(bad)) { bad = true; break; }
    umma::fence_after_sync();

    // epilogue: y of step t = tid, then the state row n = tid
    const float eo = ex2(cs);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float yd[32], yo[32];
      umma::tmem_ld32(tl + kColYd + half * 32, yd);
      umma::tmem_ld32(tl + kColYo + half * 32, yo);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c = half * 4 + q;
        float xv[8], zv[8], o[8];
        unpack8(lds128(s0 + kTileX + rx + c * 128), xv);
        if (GATE) unpack8(zr[c], zv);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float v = fmaf(eo, yo[q * 8 + j], yd[q * 8 + j]);
          v = fmaf(sD[c * 8 + j], xv[j], v);
          if (GATE) v *= silu(zv[j]);
          o[j] = in ? v : 0.f;
        }
        if (t < L) *reinterpret_cast<uint4*>(yg + row * Dm + h * P + c * 8) = pack8(o);
      }
    }
    const float etot = ex2(tot);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float ds[32];
      umma::tmem_ld32(tl + kColDS + half * 32, ds);
#pragma unroll
      for (int j = 0; j < 32; ++j) S[half * 32 + j] = fmaf(etot, S[half * 32 + j], ds[j]);
    }
    umma::fence_before_sync();
    __syncthreads();
  }

  if (bad) {
    if (tid == 0) atomicOr(p.err, kErrSsdWait);
    umma::mbar_wait(bar, phase ^ 1u, kSsdWaitLimit);  // the products still in flight, bounded
  } else if (p.h_final) {
#pragma unroll
    for (int j = 0; j < P; ++j) p.h_final[((b * Dm + h * P + j) * N) + tid] = S[j];
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 0) umma::tmem_dealloc(tm, kTmemCols);
}

template <bool GATE>
cudaError_t launch_g(const SsdParams& p, cudaStream_t s) {
  auto* k = ssd_kernel<GATE>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  const int64_t grid = p.batch * p.nheads;
  k<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t ssd_smem_bytes() { return kSmemBytes; }

cudaError_t launch_ssd(const SsdParams& p, cudaStream_t s) {
  if (p.headdim != P || p.dstate != N || p.batch * p.nheads <= 0 ||
      p.batch * p.nheads > 0x7FFFFFFF)
    return cudaErrorInvalidValue;
  return p.z ? launch_g<true>(p, s) : launch_g<false>(p, s);
}

}  // namespace ssm
