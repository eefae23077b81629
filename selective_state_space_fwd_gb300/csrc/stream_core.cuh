// stream_core.cuh -- the STREAM tier's kernel template: a channel-pair register sweep.
//
// Work split.  Every (b, d, n) recurrence h_t = Abar_t h_{t-1} + b_t is
// independent across channels and states ([P1] s1.1 "channel parallelism");
// when batch * dim * dstate fills the GPU, the cheapest schedule runs each
// recurrence serially in time in registers and spends no instructions on
// combining partial scans.  A lane owns R consecutive channels times G
// consecutive states; NG = N / G lanes share a channel group and a warp covers
// CW = (32 / NG) * R channels.  Per step and (channel, state) the work is one
// MUFU ex2 and four fp32 operations (delta*A, delta*x*B, the state update, the
// C contraction), issued as f32x2 instructions over PAIRS OF CHANNELS: the
// per-channel operands (delta, delta*x, the state) come straight from the
// vector loads and the per-state operands (B_n, C_n) are shared by the pair.
// Holding R channels makes every B/C value a lane loads serve R channels and
// every delta/x value serve G states, which is what bounds the shared-memory
// to register traffic per (channel, state).  The C contraction is a sum over
// the NG lanes of a channel group: each lane stores its per-step partial sums
// to a per-warp shared buffer, and every 16 steps an epilogue sums the NG
// partials of each (step, channel), adds the D residual, applies the silu(z)
// gate and stores y ([P1] s3.3: everything between the loads of x, delta, B,
// C and the store of y is fused; h never leaves registers).
//
// Data movement.  A CTA covers W warps (chosen at launch) of CW consecutive
// channels of one batch row.  Time is cut into tiles of T steps; per tile TMA
// copies each warp's x, delta (and z) slab [T x CW] and the B, C rows [T x N]
// into one slot of a ring ([P1] s3.2: time is the slowest dimension, channels
// and states contiguous, so every copy is a dense box).  mbarriers with
// bounded waits order the copies and their reuse.  Boxes that run past L or D
// are zero-filled by the copy engine, and a zero delta is the identity step
// (a = 2^0 = 1, b = 0), so ragged tails need no branch ([P1] s2.3); steps of
// a loaded tile past valid_len are zeroed in shared memory the same way.
// Tiles that lie entirely past valid_len[b] are never loaded: y there is
// written as exact zeros and the state stays frozen.
#pragma once

#include <cuda.h>

#include <type_traits>

#include "common.cuh"
#include "tiers.h"

namespace ssm {
namespace stream {

typedef unsigned long long u64;
constexpr unsigned kWaitLimit = 1u << 24;  // try_wait polls before a wait gives up
constexpr unsigned kErrWait = 1u;

// ---- paired fp32: two channels per instruction ---------------------------------
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
__device__ __forceinline__ u64 add2(u64 a, u64 b) {
  u64 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ---- shared memory, mbarriers, TMA ---------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false after `limit` unsuccessful polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          unsigned limit = kWaitLimit) {
  for (unsigned i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}

// ---- tile element access ---------------------------------------------------------
// pairs<PR>: 2 PR consecutive activations (R channels of one step) as fp32 pairs.
// row<G>:    G values of a B or C row (16-byte chunks in a per-lane order), widened to fp32.
// put<R>:    R consecutive outputs to global memory (rounded for bf16).
template <typename IO> struct Tile;
template <> struct Tile<float> {
  static constexpr int kBytes = 4;
  template <int PR>
  static __device__ __forceinline__ void pairs(const float* p, u64 (&o)[PR]) {
    if constexpr (PR == 2) {
      const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(p);
      o[0] = v.x;
      o[1] = v.y;
    } else {
      static_assert(PR == 1, "one or two channel pairs per lane");
      o[0] = *reinterpret_cast<const u64*>(p);
    }
  }
  // row<G>: 16-byte chunk k of the registers comes from p + coff[k] (elements)
  template <int G>
  static __device__ __forceinline__ void row(const float* p, float (&o)[G], const int* coff) {
    if constexpr (G % 4 == 0) {
#pragma unroll
      for (int k = 0; k < G / 4; ++k) {
        const float4 v = *reinterpret_cast<const float4*>(p + coff[k]);
        o[4 * k] = v.x;
        o[4 * k + 1] = v.y;
        o[4 * k + 2] = v.z;
        o[4 * k + 3] = v.w;
      }
    } else {
      static_assert(G == 2, "2, 4, 8 or 16 states per lane");
      const float2 v = *reinterpret_cast<const float2*>(p);
      o[0] = v.x;
      o[1] = v.y;
    }
  }
  // Predicated vector store (no branch: the steps around it stay in one block
  // for the scheduler).
  template <int R>
  static __device__ __forceinline__ void put(float* p, const float (&v)[R], bool on) {
    if constexpr (R == 4)
      asm volatile(
          "{\n .reg .pred q;\n setp.ne.b32 q, %5, 0;\n"
          " @q st.global.v4.f32 [%0], {%1, %2, %3, %4};\n}\n" ::"l"(p),
          "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "r"(int(on)));
    else
      asm volatile(
          "{\n .reg .pred q;\n setp.ne.b32 q, %3, 0;\n"
          " @q st.global.v2.f32 [%0], {%1, %2};\n}\n" ::"l"(p),
          "f"(v[0]), "f"(v[1]), "r"(int(on)));
  }
  static __device__ __forceinline__ void put_zero(float* p, int64_t i) { p[i] = 0.f; }
};
template <> struct Tile<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  static __device__ __forceinline__ float lo(uint32_t w) { return __uint_as_float(w << 16); }
  static __device__ __forceinline__ float hi(uint32_t w) {
    return __uint_as_float(w & 0xffff0000u);
  }
  static __device__ __forceinline__ u64 widen(uint32_t w) { return pk2(lo(w), hi(w)); }
  template <int PR>
  static __device__ __forceinline__ void pairs(const __nv_bfloat16* p, u64 (&o)[PR]) {
    if constexpr (PR == 2) {
      const uint2 v = *reinterpret_cast<const uint2*>(p);
      o[0] = widen(v.x);
      o[1] = widen(v.y);
    } else {
      static_assert(PR == 1, "one or two channel pairs per lane");
      o[0] = widen(*reinterpret_cast<const uint32_t*>(p));
    }
  }
  template <int G>
  static __device__ __forceinline__ void row(const __nv_bfloat16* p, float (&o)[G],
                                             const int* coff) {
    if constexpr (G % 8 == 0) {
#pragma unroll
      for (int k = 0; k < G / 8; ++k) {
        const uint4 v = *reinterpret_cast<const uint4*>(p + coff[k]);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          o[8 * k + 2 * j] = lo(w[j]);
          o[8 * k + 2 * j + 1] = hi(w[j]);
        }
      }
    } else if constexpr (G == 4) {
      const uint2 v = *reinterpret_cast<const uint2*>(p);
      o[0] = lo(v.x);
      o[1] = hi(v.x);
      o[2] = lo(v.y);
      o[3] = hi(v.y);
    } else {
      static_assert(G == 2, "2, 4, 8 or 16 states per lane");
      const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
      o[0] = lo(w);
      o[1] = hi(w);
    }
  }
  template <int R>
  static __device__ __forceinline__ void put(__nv_bfloat16* p, const float (&v)[R], bool on) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
    const uint32_t wa = *reinterpret_cast<const uint32_t*>(&a);
    if constexpr (R == 4) {
      const __nv_bfloat162 c = __floats2bfloat162_rn(v[2], v[3]);
      const uint32_t wc = *reinterpret_cast<const uint32_t*>(&c);
      asm volatile(
          "{\n .reg .pred q;\n setp.ne.b32 q, %3, 0;\n"
          " @q st.global.v2.b32 [%0], {%1, %2};\n}\n" ::"l"(p),
          "r"(wa), "r"(wc), "r"(int(on)));
    } else {
      asm volatile(
          "{\n .reg .pred q;\n setp.ne.b32 q, %2, 0;\n"
          " @q st.global.b32 [%0], %1;\n}\n" ::"l"(p), "r"(wa), "r"(int(on)));
    }
  }
  static __device__ __forceinline__ void put_zero(__nv_bfloat16* p, int64_t i) {
    p[i] = __float2bfloat16_rn(0.f);
  }
};

// Shared-memory bank check for one access phase of a warp: lanes [l0, l0 + n)
// each touching R consecutive floats at offset(lane); true if no two lanes
// share a bank (32 banks of 4 bytes).  An access of R floats per lane is
// served in phases of 32 / R lanes.
template <class F>
constexpr bool phase_ok(int l0, int n, int R, F offset) {
  bool used[32] = {};
  for (int l = l0; l < l0 + n; ++l)
    for (int i = 0; i < R; ++i) {
      const int bank = (offset(l) + i) % 32;
      if (used[bank]) return false;
      used[bank] = true;
    }
  return true;
}
// Lane layout of the recurrence: lane l holds state group lane_sg of channel
// group lane_cg.  With two channels per lane the two lanes of each pair share
// a state group, so that a warp's loads of its B and C slices (16 or 8 bytes
// per lane) cost half the shared-memory wavefronts of the layout whose
// neighbouring lanes read different slices (measured on GB300: 2 against 4 for
// 16-byte loads), while the delta and x loads of the channel groups keep their
// single-pass cost.  With four channels per lane that layout would need a
// partial buffer over its size limit to stay free of bank conflicts, so those
// shapes keep state groups in consecutive lanes.
__host__ __device__ constexpr int lane_sg(int l, int NG, int R) {
  return R == 2 ? (l >> 1) % NG : l % NG;
}
__host__ __device__ constexpr int lane_cg(int l, int NG, int R) {
  return R == 2 ? (l / (2 * NG)) * 2 + (l & 1) : l / NG;
}
// The layout gives each (channel group, state group) of a warp to exactly one lane.
constexpr bool lane_layout_ok(int NG, int R) {
  bool seen[32] = {};
  for (int l = 0; l < 32; ++l) {
    const int sg = lane_sg(l, NG, R), cg = lane_cg(l, NG, R);
    if (sg < 0 || sg >= NG || cg < 0 || cg >= 32 / NG) return false;
    if (seen[cg * NG + sg]) return false;
    seen[cg * NG + sg] = true;
  }
  return true;
}

// Stride (floats) between the state groups of a partial row: compute lane l
// writes R floats at lane_sg * PS + lane_cg * R.
constexpr int pad_ps(int NG, int CW, int R) {
  for (int pad = 0; pad < 32; pad += 4) {
    const int ps = CW + pad;
    bool ok = true;
    for (int l0 = 0; l0 < 32; l0 += 32 / R)
      ok = ok && phase_ok(l0, 32 / R, R, [&](int l) {
             return lane_sg(l, NG, R) * ps + lane_cg(l, NG, R) * R;
           });
    if (ok) return ps;
  }
  return CW;
}
// Stride (floats) between the steps of the partial buffer: epilogue lane
// (cp = lane % CG, sl = lane / CG) reads R floats at sl * PROW + g * PS + cp * R.
constexpr int pad_prow(int NG, int CW, int R, int PS) {
  const int CG = 32 / NG;
  for (int pad = 0; pad < 64; pad += 4) {
    const int pr = NG * PS + pad;
    bool ok = true;
    for (int l0 = 0; l0 < 32; l0 += 32 / R)
      ok = ok && phase_ok(l0, 32 / R, R, [&](int l) { return (l / CG) * pr + (l % CG) * R; });
    if (ok) return pr;
  }
  return NG * PS;
}

// Compile-time shape of one STREAM instance.
template <int N_, int G_, int R_, typename IO_, bool GATE_, bool DTP_ = false, bool AGG_ = false,
          bool RANK_ = false>
struct Cfg {
  static constexpr int N = N_, G = G_, R = R_;
  static constexpr bool GATE = GATE_;
  // AGG: the aggregate pass of the time split -- the state recurrence only
  // (no C, no y), from a zero state for segments >= 1; writes each segment's
  // end state and its sum of delta.
  static constexpr bool AGG = AGG_;
  // DTP: the fused step-size preparation (bias, softplus, clipping) runs once
  // per tile over the warp's delta slab; for fp32 in place, for bf16 into an
  // fp32 slab of the warp (the prepared step is not rounded to bf16).
  static constexpr bool DTP = DTP_;
  // RANK: the batch rows have valid lengths and are handed to the CTAs
  // longest first (rows_ranked, row_of_rank in common.cuh)
  static constexpr bool RANK = RANK_;
  using IO = IO_;
  static constexpr int PR = R / 2;           // channel pairs per lane
  static constexpr int NG = N / G;           // lanes per channel group
  static constexpr int CG = 32 / NG;         // channel groups per warp
  static constexpr int CW = CG * R;          // channels per warp
  static constexpr int T = 64;               // steps per tile
  static constexpr int ES = Tile<IO>::kBytes;
  // steps per batch: a batch's inputs are loaded two batches ahead and its
  // decays and input terms formed one batch ahead of its recurrence
  static constexpr int U = R * G <= 8 ? 2 : 1;
  static constexpr int M = 16;                 // steps per block of the tile loop
  // per-warp buffer of the C h partial sums of one block: [M][NG][PS] floats
  // (row j: step j of the block, then state group, then channel), with the
  // paddings PS - CW and PROW - NG PS chosen so that the compute lanes'
  // writes and the epilogue lanes' reads hit distinct banks
  static constexpr int PS = pad_ps(NG, CW, R);
  static constexpr int PROW = pad_prow(NG, CW, R, PS);
  static constexpr int PBYTES = M * PROW * 4;
  static constexpr bool DSF = DTP && ES == 2;          // the fp32 delta slab exists
  static constexpr int DSFBYTES = DSF ? T * CW * 4 : 0;
  using DT = typename std::conditional<DSF, float, IO>::type;  // delta as the lanes read it
  static constexpr int NACT = GATE ? 3 : 2;    // activation tensors per tile
  // A lane's slice of a B or C row is MCH 16-byte chunks of CHUNK elements.
  // The lanes of one access phase start their slices 16 * MCH bytes apart, so
  // for MCH > 1 they would collide in the banks; each lane therefore visits
  // its chunks rotated by ROT(sg) and keeps its states in that order.
  static constexpr int CHUNK = 16 / ES;
  static constexpr int MCH = G * ES >= 16 ? G * ES / 16 : 1;
  static constexpr int SLAB = T * CW * ES;     // one warp's [T x CW] tile of one tensor
  static constexpr int ROWT = T * N * ES;      // [T x N] tile of B or C
  static_assert(R == 2 || R == 4, "two or four channels per lane");
  static_assert(lane_layout_ok(NG, R), "lane layout");
  static_assert(G >= 2 && N % G == 0 && NG <= 16 && (NG & (NG - 1)) == 0, "state groups");
  static_assert((CW * ES) % 16 == 0 && (N * ES) % 16 == 0, "TMA box rows are 16-byte multiples");
  static_assert(T % M == 0 && M % (2 * U) == 0 && M % NG == 0, "tile steps");
  static_assert(PROW % 4 == 0 && PS % 4 == 0 && PBYTES <= 12 * 1024, "partial buffer");
  static_assert(SLAB % 128 == 0 && ROWT % 128 == 0, "slot alignment");
  static_assert(!(AGG && (DTP || GATE)), "the aggregate pass takes delta as given and has no gate");
  static_assert(!(AGG && RANK), "the aggregate pass runs segments, not ranked rows");
};

// One batch of U steps' inputs for this lane, as loaded from the tile.
template <class K>
struct Raw {
  u64 dt[K::U][K::PR], x[K::U][K::PR];
  float b[K::U][K::G], c[K::U][K::G];
};

template <class K>
__device__ __forceinline__ void load_batch(Raw<K>& r, const typename K::DT* ds,
                                           const typename K::IO* xs, const typename K::IO* bs,
                                           const typename K::IO* cs, int s, const int* coff) {
  using TL = Tile<typename K::IO>;
#pragma unroll
  for (int u = 0; u < K::U; ++u) {
    Tile<typename K::DT>::template pairs<K::PR>(ds + (s + u) * K::CW, r.dt[u]);
    TL::template pairs<K::PR>(xs + (s + u) * K::CW, r.x[u]);
    TL::template row<K::G>(bs + (s + u) * K::N, r.b[u], coff);
    if constexpr (!K::AGG) TL::template row<K::G>(cs + (s + u) * K::N, r.c[u], coff);
  }
}

// One batch of U steps, ready for the recurrence: the decays Abar = exp(delta A)
// ([P1] s2.4: 2^(delta * A log2 e), one MUFU ex2 each), the input terms
// b = delta B x ([P1] s3.3), per channel pair and state; the C values.
template <class K>
struct Prep {
  u64 ab[K::U][K::PR][K::G], bi[K::U][K::PR][K::G];
  float c[K::U][K::G];
  u64 dt[K::AGG ? K::U : 1][K::PR];  // the aggregate pass sums delta
};

template <class K>
__device__ __forceinline__ void prepare(Prep<K>& o, const Raw<K>& r, const u64 (&a2)[K::PR][K::G]) {
#pragma unroll
  for (int u = 0; u < K::U; ++u) {
#pragma unroll
    for (int q = 0; q < K::PR; ++q) {
      const u64 dt = r.dt[u][q];
      if constexpr (K::AGG) o.dt[u][q] = dt;
      const u64 ux = mul2(dt, r.x[u][q]);  // delta x
#pragma unroll
      for (int n = 0; n < K::G; ++n) {
        const float2 arg = upk2(mul2(dt, a2[q][n]));
        o.ab[u][q][n] = pk2(ex2(arg.x), ex2(arg.y));
        o.bi[u][q][n] = mul2(ux, pk2(r.b[u][n], r.b[u][n]));
      }
    }
    if constexpr (!K::AGG) {
#pragma unroll
      for (int n = 0; n < K::G; ++n) o.c[u][n] = r.c[u][n];
    }
  }
}

// Kernel arguments besides the tensor maps.
struct LaunchArgs {
  int warps;       // W, warps per CTA
  int stages;      // slots in the ring
  int stage_bytes;
  unsigned int* err;  // sticky error word
};

template <class K>
__global__ void __launch_bounds__(128, 1)
    stream_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dt,
                  const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_b,
                  const __grid_constant__ CUtensorMap tm_c, const ScanParams p,
                  const LaunchArgs la) {
  using IO = typename K::IO;
  using TL = Tile<IO>;
  constexpr int N = K::N, G = K::G, R = K::R, PR = K::PR, NG = K::NG, CW = K::CW;
  constexpr int T = K::T, U = K::U, M = K::M, CG = K::CG;
  extern __shared__ __align__(128) char smem[];
  const int W = la.warps, STAGES = la.stages, SB = la.stage_bytes;
  // this warp's partial-sum buffer, after the ring
  float* pbuf = reinterpret_cast<float*>(smem + STAGES * SB + (threadIdx.x >> 5) * K::PBYTES);
  float* dsf = reinterpret_cast<float*>(smem + STAGES * SB + W * K::PBYTES +
                                        (threadIdx.x >> 5) * K::DSFBYTES);  // fp32 delta slab
  uint64_t* full =
      reinterpret_cast<uint64_t*>(smem + STAGES * SB + W * (K::PBYTES + K::DSFBYTES));
  uint64_t* empty = full + STAGES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cpc = W * CW;
  const int64_t n_cb = (p.dim + cpc - 1) / cpc;
  // (batch row, segment of the time split); ranked instances take the rows
  // longest first
  const int64_t row = K::RANK && p.n_seg == 1 && rows_ranked(p)
                          ? row_of_rank(p, blockIdx.x / n_cb)
                          : blockIdx.x / n_cb;
  const int64_t b = row / p.n_seg;
  const int seg = static_cast<int>(row % p.n_seg);
  if (K::AGG && seg == p.n_seg - 1) return;  // the last segment's aggregate is not needed
  const int d0 = static_cast<int>((blockIdx.x % n_cb) * cpc);
  const int cg = lane_cg(lane, NG, R), sg = lane_sg(lane, NG, R);
  const int dw = d0 + warp * CW;       // the warp's first channel
  const int64_t dl = dw + cg * R;      // the lane's first channel
  const bool d_ok = dl < p.dim;        // all R channels valid (dim is a multiple of R)
  const int64_t L = p.seqlen;
  // this CTA's steps: [seg0, seg0 + Ls) of the row, lv of them valid
  const int64_t seg0 = p.seg_len > 0 ? seg * p.seg_len : 0;
  const int64_t Ls = p.seg_len > 0 ? min(p.seg_len, L - seg0) : L;
  const int64_t lv = min(max(valid_steps(p, b) - seg0, int64_t(0)), Ls);
  const int n_tiles = static_cast<int>((lv + T - 1) / T);  // tiles with a valid step
  const bool producer = threadIdx.x == 0;

  auto issue = [&](int tile, int slot) {
    char* st = smem + slot * SB;
    const int t0 = static_cast<int>(seg0) + tile * T;
    mbar_expect_tx(&full[slot], K::AGG ? SB - K::ROWT : SB);
    for (int w = 0; w < W; ++w) {
      tma_load_3d(st + (0 * W + w) * K::SLAB, &tm_x, d0 + w * CW, t0, static_cast<int>(b),
                  &full[slot]);
      tma_load_3d(st + (1 * W + w) * K::SLAB, &tm_dt, d0 + w * CW, t0, static_cast<int>(b),
                  &full[slot]);
      if constexpr (K::GATE)
        tma_load_3d(st + (2 * W + w) * K::SLAB, &tm_z, d0 + w * CW, t0, static_cast<int>(b),
                    &full[slot]);
    }
    char* rows = st + K::NACT * W * K::SLAB;
    tma_load_3d(rows, &tm_b, 0, t0, static_cast<int>(b), &full[slot]);
    if constexpr (!K::AGG) tma_load_3d(rows + K::ROWT, &tm_c, 0, t0, static_cast<int>(b), &full[slot]);
  };

  if (producer) {
    for (int st = 0; st < STAGES; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], W);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (producer)
    for (int st = 0; st < STAGES && st < n_tiles; ++st) issue(st, st);

  // Register n of a lane holds state gsn(n) of its channels (chunk rotation,
  // see Cfg::MCH); coff[k] is the row offset of the lane's k-th loaded chunk.
  constexpr int CHK = K::CHUNK, MCH = K::MCH;
  const int rot = MCH > 1 ? (sg / (8 / MCH)) % MCH : 0;
  int coff[MCH];
#pragma unroll
  for (int k = 0; k < MCH; ++k) coff[k] = ((k + rot) % MCH) * CHK;
  auto gsn = [&](int n) {
    return MCH > 1 ? sg * G + ((n / CHK + rot) % MCH) * CHK + n % CHK : sg * G + n;
  };
  // Per-lane constants: log2(e)-scaled A for (channel pair, state), the
  // initial state: the caller's h0 for the first segment; for a later one the
  // state carried into it (the aggregate pass starts those from zero).
  const float* h0row = seg == 0 ? (p.h0 ? p.h0 + b * p.dim * N : nullptr)
                                : (!K::AGG && p.seg_h0 ? p.seg_h0 + row * p.dim * N : nullptr);
  u64 a2[PR][G], h2[PR][G];
#pragma unroll
  for (int q = 0; q < PR; ++q) {
    const int64_t d_lo = dl + 2 * q, d_hi = d_lo + 1;
#pragma unroll
    for (int n = 0; n < G; ++n) {
      float lo = 0.f, hi = 0.f;
      if (d_ok) {
        lo = __ldg(p.A + d_lo * N + gsn(n)) * kLog2e;
        hi = __ldg(p.A + d_hi * N + gsn(n)) * kLog2e;
      }
      a2[q][n] = pk2(lo, hi);
      float h_lo = 0.f, h_hi = 0.f;  // [P1] s4.1: h_0 = 0 unless given
      if (d_ok && h0row) {
        h_lo = __ldg(h0row + d_lo * N + gsn(n));
        h_hi = __ldg(h0row + d_hi * N + gsn(n));
      }
      h2[q][n] = pk2(h_lo, h_hi);
    }
  }

  u64 dsum[PR];  // the aggregate pass: sum of delta of the lane's channels
#pragma unroll
  for (int q = 0; q < PR; ++q) dsum[q] = 0;
  // Bias of the channels this lane prepares step sizes for (element e of the
  // warp's slab belongs to channel e % CW; lane l visits e = l + 32 k).
  constexpr int NBV = CW > 32 ? CW / 32 : 1;
  float dbias[NBV];
#pragma unroll
  for (int i = 0; i < NBV; ++i) {
    const int c = (lane + 32 * i) % CW;
    dbias[i] = (K::DTP && dw + c < p.dim) ? delta_bias(p.dt_bias, dw + c) : 0.f;
  }
  // The epilogue's view of the warp: lane (cp, sl) finishes the outputs of
  // channels dw + cp R .. + R at steps sl, sl + NG, ... of each block.
  const int cp = lane % CG, sl = lane / CG;
  const int64_t de = dw + cp * R;
  const bool de_ok = de < p.dim;
  u64 dsk[PR];  // D residual of the epilogue's channels
#pragma unroll
  for (int q = 0; q < PR; ++q)
    dsk[q] = (de_ok && p.D) ? pk2(__ldg(p.D + de + 2 * q), __ldg(p.D + de + 2 * q + 1)) : 0;
  IO* __restrict__ yout = static_cast<IO*>(p.y);
  const bool want_states = !K::AGG && p.states != nullptr;
  // Chunk c ends at step min((c+1) chunk_len, L) - 1 ([P1] s3.4).
  auto chunk_end = [&](int64_t c) { return min((c + 1) * p.chunk_len, L) - 1; };
  int64_t next_c = want_states ? seg0 / p.chunk_len : 0;  // first chunk ending in the segment
  int64_t next_ce = want_states ? chunk_end(next_c) : INT64_MAX;
  // the lane's G states of each of its R channels, as rows of `dst`
  auto put_state = [&](float* dst) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float v[G];
#pragma unroll
      for (int n = 0; n < G; ++n) {
        const float2 hv = upk2(h2[r / 2][n]);
        v[n] = (r & 1) ? hv.y : hv.x;
      }
      float* row = dst + (dl + r) * N;
      if constexpr (G % 4 == 0) {  // 4 consecutive registers are 4 consecutive states
#pragma unroll
        for (int k = 0; k < G / 4; ++k)
          *reinterpret_cast<float4*>(row + gsn(4 * k)) =
              make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
      } else {
        reinterpret_cast<float2*>(row + sg * G)[0] = make_float2(v[0], v[1]);
      }
    }
  };
  auto store_state = [&](int64_t t) {
    if (d_ok) put_state(p.states + (b * p.n_chunks + t / p.chunk_len) * p.dim * N);
  };

  bool ok = true;
  for (int i = 0; i < n_tiles && ok; ++i) {
    const int slot = i % STAGES;
    char* st = smem + slot * SB;
    ok = mbar_wait(&full[slot], (i / STAGES) & 1);
    if (!ok) break;
    // refill the slot freed by the previous tile (every warp is done with it)
    if (producer && i >= 1 && i - 1 + STAGES < n_tiles) {
      const int ps = (i - 1) % STAGES;
      ok = mbar_wait(&empty[ps], ((i - 1) / STAGES) & 1);
      if (ok) issue(i - 1 + STAGES, ps);
    }
    const IO* xw = reinterpret_cast<const IO*>(st + (0 * W + warp) * K::SLAB);  // warp's slabs
    const IO* zw = reinterpret_cast<const IO*>(st + (2 * W + warp) * K::SLAB);
    const IO* xs = xw + cg * R;  // this lane's channels
    IO* dslab = reinterpret_cast<IO*>(st + (1 * W + warp) * K::SLAB);  // warp's delta slab
    const typename K::DT* ds;  // this lane's delta column, as the recurrence reads it
    const IO* bs = reinterpret_cast<const IO*>(st + K::NACT * W * K::SLAB) + sg * G;
    const IO* cs = bs + T * N;
    const int64_t tl = static_cast<int64_t>(i) * T;                 // tile start in the segment
    const int64_t t0 = seg0 + tl;                                    // tile start in the row
    const int steps = static_cast<int>(lv - tl < T ? lv - tl : T);  // valid steps in tile
    IO* ybase = yout + (b * L + t0) * p.dim + de;                    // y[b, t0, de]
    if constexpr (K::DTP) {
      // The step size of every (step, channel) of the warp, prepared once:
      // delta + dt_bias[d], softplus, clipping ([P1] s3.3).  Rows past the
      // valid steps and channels past dim become 0 (identity steps).
      typename K::DT* dst;
      if constexpr (K::DSF) dst = dsf;
      else dst = dslab;
      // groups of 8 elements per lane: loads, then arithmetic, then stores, so
      // that the in-place update of fp32 slabs does not serialise the loads
      constexpr int PER = T * CW / 32, GRP = 8;
      static_assert(PER % GRP == 0, "delta preparation groups");
#pragma unroll
      for (int g0 = 0; g0 < PER; g0 += GRP) {
        float v[GRP];
#pragma unroll
        for (int k = 0; k < GRP; ++k) {
          const int e = lane + 32 * (g0 + k);
          if constexpr (K::ES == 2) v[k] = __bfloat162float(dslab[e]);
          else v[k] = dslab[e];
        }
#pragma unroll
        for (int k = 0; k < GRP; ++k) {
          const int e = lane + 32 * (g0 + k);
          const int row = e / CW, c = e % CW;
          const float pv = prep_delta(v[k], dbias[(g0 + k) % NBV], p);
          v[k] = (row < steps && dw + c < p.dim) ? pv : 0.f;
        }
#pragma unroll
        for (int k = 0; k < GRP; ++k) dst[lane + 32 * (g0 + k)] = typename K::DT(v[k]);
      }
      ds = dst + cg * R;
      __syncwarp();
    } else {
      ds = dslab + cg * R;
    }
    if (steps < T) {
      // Steps of the tile past valid_len become the identity (a = 1, b = 0,
      // [P1] s2.3): their delta, x, B and C are set to zero in the tile, so
      // no per-step test is needed and padded values never reach the state.
      // The B and C rows are shared by the CTA's warps: each warp zeroes them
      // itself (every writer stores the same zeros, and a warp reads them only
      // after its own pass), so no CTA-wide barrier is needed.
      IO* dsw = dslab;
      IO* xsw = const_cast<IO*>(xw);
      for (int e = steps * CW + lane; e < T * CW; e += 32) {
        dsw[e] = IO(0.f);
        xsw[e] = IO(0.f);
      }
      IO* rows = reinterpret_cast<IO*>(st + K::NACT * W * K::SLAB);
      for (int e = steps * N + lane; e < T * N; e += 32) {
        rows[e] = IO(0.f);          // B
        rows[T * N + e] = IO(0.f);  // C
      }
      __syncwarp();
    }

    // Epilogue of the block starting at step s0 of the tile: sum the NG
    // partials of each (step, channel), add D x, gate, store.  Every lane's
    // items are independent, so their shared-memory latencies overlap.
    auto epilogue = [&](int s0) {
      __syncwarp();
#pragma unroll
      for (int i = 0; i < M / NG; ++i) {
        const int j = sl + NG * i;  // step within the block
        const int so = s0 + j;      // step within the tile
        const float* pr = pbuf + j * K::PROW + cp * R;
        u64 sum[PR];
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          u64 part[PR];
          Tile<float>::template pairs<PR>(pr + g * K::PS, part);
#pragma unroll
          for (int q = 0; q < PR; ++q) sum[q] = g == 0 ? part[q] : add2(sum[q], part[q]);
        }
        u64 xq[PR];
        TL::template pairs<PR>(xw + so * CW + cp * R, xq);
        float o[R];
#pragma unroll
        for (int q = 0; q < PR; ++q) {
          const float2 yv = upk2(fma2(dsk[q], xq[q], sum[q]));  // + D x
          o[2 * q] = yv.x;
          o[2 * q + 1] = yv.y;
        }
        if constexpr (K::GATE) {
          u64 zq[PR];
          TL::template pairs<PR>(zw + so * CW + cp * R, zq);
#pragma unroll
          for (int q = 0; q < PR; ++q) {
            const float2 zz = upk2(zq[q]);
            o[2 * q] *= silu(zz.x);  // * silu(z)
            o[2 * q + 1] *= silu(zz.y);
          }
        }
        TL::template put<R>(ybase + static_cast<int64_t>(so) * p.dim, o, de_ok && so < steps);
      }
      __syncwarp();
    };

    // Software pipeline over batches of U steps: while batch k runs its
    // recurrence (the fp32 pipe), the decays and input terms of batch k+1 are
    // formed (the MUFU pipe) and the loads of batch k+2 are in flight.  A
    // block of M steps holds an even number of batches, so the roles of the
    // two raw and two prepared buffers are fixed at compile time.
    Raw<K> raw[2];
    Prep<K> prep[2];
    load_batch<K>(raw[0], ds, xs, bs, cs, 0, coff);
    load_batch<K>(raw[1], ds, xs, bs, cs, U & (T - 1), coff);
    prepare<K>(prep[0], raw[0], a2);
    for (int s0 = 0; s0 < steps; s0 += M) {
      const int64_t b_last = t0 + s0 + M - 1;  // the block's last step
      // CHECK: a chunk ends strictly inside the block, test every step (a
      // branch per step would keep the compiler from overlapping steps).
      auto run_block = [&](auto check) {
        constexpr bool CHECK = decltype(check)::value;
#pragma unroll
        for (int k = 0; k < M / U; ++k) {
          const int s = s0 + k * U;
          prepare<K>(prep[(k + 1) & 1], raw[(k + 1) & 1], a2);  // batch k+1
          // batch k+2; near the tile's end this wraps to its start (unused)
          load_batch<K>(raw[k & 1], ds, xs, bs, cs, (s + 2 * U) & (T - 1), coff);
          const Prep<K>& cur = prep[k & 1];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int j = k * U + u;  // step within the block
            if constexpr (K::AGG) {  // the state only, and the sum of delta
#pragma unroll
              for (int q = 0; q < PR; ++q) {
                dsum[q] = add2(dsum[q], cur.dt[u][q]);
#pragma unroll
                for (int n = 0; n < G; ++n)
                  h2[q][n] = fma2(cur.ab[u][q][n], h2[q][n], cur.bi[u][q][n]);  // h = Abar h + b
              }
              continue;
            }
            // C h accumulates in NA independent chains (short dependency
            // chains: one warp per scheduler has little else to overlap)
            constexpr int NA = G >= 8 ? 4 : (G >= 4 ? 2 : 1);
            u64 acc[NA][PR];
#pragma unroll
            for (int n = 0; n < G; ++n) {
              const u64 cc = pk2(cur.c[u][n], cur.c[u][n]);
#pragma unroll
              for (int q = 0; q < PR; ++q) {
                h2[q][n] = fma2(cur.ab[u][q][n], h2[q][n], cur.bi[u][q][n]);  // h = Abar h + b
                if (n < NA)
                  acc[n][q] = mul2(cc, h2[q][n]);
                else
                  acc[n % NA][q] = fma2(cc, h2[q][n], acc[n % NA][q]);  // C h
              }
            }
            // this lane's partial of sum_n C_n h_n, to the block's buffer
            u64 part[PR];
#pragma unroll
            for (int q = 0; q < PR; ++q) {
#pragma unroll
              for (int a = NA / 2; a >= 1; a /= 2)
#pragma unroll
                for (int i = 0; i < a; ++i) acc[i][q] = add2(acc[i][q], acc[i + a][q]);
              part[q] = acc[0][q];
            }
            float* pw = pbuf + j * K::PROW + sg * K::PS + cg * R;
            if constexpr (PR == 2)
              *reinterpret_cast<ulonglong2*>(pw) = make_ulonglong2(part[0], part[1]);
            else
              *reinterpret_cast<u64*>(pw) = part[0];
            if constexpr (CHECK) {
              if (t0 + s + u == next_ce) {  // [P1] s3.4 chunk boundary state
                store_state(next_ce);
                ++next_c;
                next_ce = next_c < p.n_chunks ? chunk_end(next_c) : INT64_MAX;
              }
            }
          }
        }
      };
      if (next_ce < b_last)
        run_block(std::true_type{});
      else
        run_block(std::false_type{});
      if (next_ce == b_last) {  // a chunk ends with the block
        store_state(next_ce);
        ++next_c;
        next_ce = next_c < p.n_chunks ? chunk_end(next_c) : INT64_MAX;
      }
      if constexpr (!K::AGG) epilogue(s0);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
  if (!ok) {
    if (lane == 0) atomicOr(la.err, kErrWait);
    return;
  }

  if constexpr (K::AGG) {
    // the segment's aggregate: its end state from a zero start (or the
    // caller's h0 for the first segment) and its sum of delta over the valid
    // steps (padded steps have delta 0)
    if (d_ok) {
      put_state(p.seg_hend + row * p.dim * N);
      if (sg == 0) {
#pragma unroll
        for (int q = 0; q < PR; ++q) {
          const float2 v = upk2(dsum[q]);
          p.seg_dtsum[row * p.dim + dl + 2 * q] = v.x;
          p.seg_dtsum[row * p.dim + dl + 2 * q + 1] = v.y;
        }
      }
    }
    return;
  }
  // Steps past valid_len: exact zeros, frozen state for the remaining chunk ends.
  if (lv < Ls) {
    const int64_t total = (Ls - lv) * CW;
    for (int64_t e = lane; e < total; e += 32) {
      const int64_t t = seg0 + lv + e / CW;
      const int c = static_cast<int>(e % CW);
      if (dw + c < p.dim) TL::put_zero(yout, (b * L + t) * p.dim + dw + c);
    }
  }
  if (want_states)  // frozen state for the chunks that end in this segment
    for (; next_c < p.n_chunks && chunk_end(next_c) < seg0 + Ls; ++next_c)
      store_state(chunk_end(next_c));
  if (p.h_final && d_ok && seg == p.n_seg - 1)
    put_state(p.h_final + b * p.dim * N);  // state after the last step
}

// Host side, defined in kernel_stream.cu.
bool make_map(CUtensorMap* m, const void* base, bool bf16, int64_t inner, int64_t L, int64_t batch,
              int box_inner, int box_t);
unsigned int* error_word();
int max_dynamic_smem();
bool tma_encode_available();  // the driver's tensor-map encoder was found

template <class K>
int stage_bytes(int warps) {
  return K::NACT * warps * K::SLAB + 2 * K::ROWT;
}

template <class K>
cudaError_t launch_k(const ScanParams& p, cudaStream_t s, int warps, int stages) {
  const bool bf16 = sizeof(typename K::IO) == 2;
  CUtensorMap mx, mdt, mz, mb, mc;
  if (!make_map(&mx, p.x, bf16, p.dim, p.seqlen, p.batch, K::CW, K::T) ||
      !make_map(&mdt, p.delta, bf16, p.dim, p.seqlen, p.batch, K::CW, K::T) ||
      !make_map(&mb, p.B, bf16, K::N, p.seqlen, p.batch, K::N, K::T) ||
      !make_map(&mc, p.C, bf16, K::N, p.seqlen, p.batch, K::N, K::T))
    return cudaErrorInvalidValue;
  if constexpr (K::GATE) {
    if (!make_map(&mz, p.z, bf16, p.dim, p.seqlen, p.batch, K::CW, K::T))
      return cudaErrorInvalidValue;
  } else {
    mz = mx;  // unused
  }
  LaunchArgs la;
  la.warps = warps;
  la.stages = stages;
  la.stage_bytes = stage_bytes<K>(warps);
  la.err = error_word();
  if (la.err == nullptr) return cudaErrorInvalidValue;
  const int smem = stages * la.stage_bytes + warps * (K::PBYTES + K::DSFBYTES) + 2 * stages * 8;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(stream_kernel<K>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         max_dynamic_smem());
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  if (smem > max_dynamic_smem()) return cudaErrorInvalidValue;
  const int64_t n_cb = (p.dim + warps * K::CW - 1) / (warps * K::CW);
  const int64_t grid = n_cb * p.batch * p.n_seg;
  stream_kernel<K><<<static_cast<unsigned>(grid), warps * 32, smem, s>>>(mx, mdt, mz, mb, mc, p,
                                                                        la);
  return cudaGetLastError();
}

// Every launcher of one (N, G, R) instance: fp32 / bf16, with / without gate.
template <int N, int G, int R>
cudaError_t launch_ngr(const ScanParams& p, bool bf16, cudaStream_t s, int warps, int stages);

// The aggregate pass of the time split (default shapes only).
template <int N, int G, int R>
cudaError_t launch_ngr_agg(const ScanParams& p, bool bf16, cudaStream_t s, int warps, int stages);

// Per-stage bytes of an instance, for the host's ring sizing.
template <int N, int G, int R>
int stage_bytes_ngr(bool bf16, bool gate, int warps);

// bf16 instances exist when the B/C rows and a warp's activation rows are at
// least 16-byte multiples (TMA boxes).
template <int N, int G, int R>
constexpr bool bf16_ok() {
  return N * 2 >= 16 && (32 / (N / G)) * R * 2 % 16 == 0;
}

template <int N, int G, int R, bool DTP, bool RANK>
cudaError_t launch_ngr_dtp(const ScanParams& p, bool bf16, cudaStream_t s, int w, int st) {
  if (bf16) {
    if constexpr (bf16_ok<N, G, R>())
      return p.z ? launch_k<Cfg<N, G, R, __nv_bfloat16, true, DTP, false, RANK>>(p, s, w, st)
                 : launch_k<Cfg<N, G, R, __nv_bfloat16, false, DTP, false, RANK>>(p, s, w, st);
    else
      return cudaErrorInvalidValue;
  }
  return p.z ? launch_k<Cfg<N, G, R, float, true, DTP, false, RANK>>(p, s, w, st)
             : launch_k<Cfg<N, G, R, float, false, DTP, false, RANK>>(p, s, w, st);
}

// Shapes compiled with the fused step-size preparation: the default ones.
constexpr bool dtp_shape(int n, int g, int r) {
  return r == 2 && ((n <= 16 && g == 4) || (n >= 32 && g == 8));
}

template <int N, int G, int R>
cudaError_t launch_ngr_impl(const ScanParams& p, bool bf16, cudaStream_t s, int w, int st) {
  // ranked instances exist for the default shapes (the host side of rows_ranked)
  const bool rank = p.valid_len != nullptr && p.batch <= 32 && p.n_seg == 1;
  if (has_delta_prep(p)) {
    if constexpr (dtp_shape(N, G, R))
      return rank ? launch_ngr_dtp<N, G, R, true, true>(p, bf16, s, w, st)
                  : launch_ngr_dtp<N, G, R, true, false>(p, bf16, s, w, st);
    else
      return cudaErrorInvalidValue;
  }
  if constexpr (dtp_shape(N, G, R))
    if (rank) return launch_ngr_dtp<N, G, R, false, true>(p, bf16, s, w, st);
  return launch_ngr_dtp<N, G, R, false, false>(p, bf16, s, w, st);
}

template <int N, int G, int R>
cudaError_t launch_ngr_agg_impl(const ScanParams& p, bool bf16, cudaStream_t s, int w, int st) {
  if constexpr (dtp_shape(N, G, R)) {
    if (bf16) {
      if constexpr (bf16_ok<N, G, R>())
        return launch_k<Cfg<N, G, R, __nv_bfloat16, false, false, true>>(p, s, w, st);
      else
        return cudaErrorInvalidValue;
    }
    return launch_k<Cfg<N, G, R, float, false, false, true>>(p, s, w, st);
  } else {
    return cudaErrorInvalidValue;
  }
}

template <int N, int G, int R>
int stage_bytes_impl(bool bf16, bool gate, int w) {
  if (bf16) {
    if constexpr (bf16_ok<N, G, R>())
      return gate ? stage_bytes<Cfg<N, G, R, __nv_bfloat16, true>>(w)
                  : stage_bytes<Cfg<N, G, R, __nv_bfloat16, false>>(w);
    else
      return 0;
  }
  return gate ? stage_bytes<Cfg<N, G, R, float, true>>(w)
              : stage_bytes<Cfg<N, G, R, float, false>>(w);
}

#define SSM_STREAM_DEFINE(N_, G_, R_)                                                        \
  template <>                                                                                \
  cudaError_t launch_ngr<N_, G_, R_>(const ScanParams& p, bool bf16, cudaStream_t s, int w, \
                                     int st) {                                               \
    return launch_ngr_impl<N_, G_, R_>(p, bf16, s, w, st);                                   \
  }                                                                                          \
  template <>                                                                                \
  cudaError_t launch_ngr_agg<N_, G_, R_>(const ScanParams& p, bool bf16, cudaStream_t s,    \
                                         int w, int st) {                                    \
    return launch_ngr_agg_impl<N_, G_, R_>(p, bf16, s, w, st);                               \
  }                                                                                          \
  template <>                                                                                \
  int stage_bytes_ngr<N_, G_, R_>(bool bf16, bool gate, int w) {                             \
    return stage_bytes_impl<N_, G_, R_>(bf16, gate, w);                                      \
  }

// Instances (N, G, R): states per lane G, channels per lane R.
#define SSM_STREAM_INSTANCES(X)                              \
  X(4, 4, 2) X(4, 4, 4)                                      \
  X(8, 4, 2) X(8, 4, 4) X(8, 8, 2)                           \
  X(16, 4, 2) X(16, 4, 4) X(16, 8, 2) X(16, 8, 4) X(16, 16, 2) \
  X(32, 4, 4) X(32, 8, 2) X(32, 8, 4)                        \
  X(64, 8, 2) X(64, 8, 4) X(64, 16, 2)

#define SSM_STREAM_DECLARE(N_, G_, R_)                                                      \
  template <>                                                                               \
  cudaError_t launch_ngr<N_, G_, R_>(const ScanParams&, bool, cudaStream_t, int, int);     \
  template <>                                                                               \
  cudaError_t launch_ngr_agg<N_, G_, R_>(const ScanParams&, bool, cudaStream_t, int, int); \
  template <>                                                                               \
  int stage_bytes_ngr<N_, G_, R_>(bool, bool, int);

}  // namespace stream
}  // namespace ssm
