// kernel_stream.cu -- the STREAM tier of libssmscan: a state-split register sweep.
//
// Work split.  Every (b, d, n) recurrence h_t = Abar_t h_{t-1} + b_t is
// independent across channels and states ([P1] s1.1 "channel parallelism");
// when batch * dim * dstate fills the GPU, the cheapest schedule is to run
// each recurrence serially in time in registers and spend no instructions on
// combining partial scans.  A lane owns G consecutive states of one channel;
// NG = N / G lanes share a channel, and a warp covers CH = 32 / NG channels.
// Per step and state the work is one MUFU ex2 and four fp32 operations
// (delta*A, delta*x*B, the state update, the C contraction), issued as paired
// f32x2 instructions: two states per instruction.  The C contraction is a sum
// over the NG lanes of a channel; it is reduced with a shuffle reduce-scatter
// once per NG steps, after which each lane owns one (step, channel) output and
// applies the D residual and the silu(z) gate ([P1] s3.3: everything between
// the loads of x, delta, B, C and the store of y is fused; h never leaves
// registers).
//
// Data movement.  A CTA covers CPC = CH * WPC consecutive channels of one
// batch row.  Time is cut into tiles of T steps; TMA copies the x, delta (and
// z) tile [T x CPC] and the B, C rows [T x N] of a tile into a ring of STAGES
// shared-memory slots ([P1] s3.2: time is the slowest dimension, channels and
// states contiguous, so every copy is a dense box).  mbarriers with bounded
// waits order the copies and their reuse.  Boxes that run past L or D are
// zero-filled by the copy engine, and a zero delta is the identity step
// (a = 2^0 = 1, b = 0), so ragged tails need no branch ([P1] s2.3).  Tiles
// that lie entirely past valid_len[b] are never loaded: y there is written as
// exact zeros and the state stays frozen.
#include <cuda.h>

#include "common.cuh"
#include "tiers.h"

namespace ssm {

// Sticky error word of the bounded waits (0 = no error).  Set with atomicOr
// by a CTA whose mbarrier wait gave up; read and cleared by the host through
// ssm_check_device_errors().
__device__ unsigned int g_stream_error = 0;

namespace {

typedef unsigned long long u64;
constexpr unsigned kWaitLimit = 1u << 24;  // try_wait polls before a wait gives up
constexpr unsigned kErrWait = 1u;

// ---- paired fp32 (two lanes of state per instruction) ----------------------
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
#ifndef SSM_SCALAR_PAIRS
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
#else  // the same arithmetic as two scalar fp32 instructions (comparison builds)
__device__ __forceinline__ u64 mul2(u64 a, u64 b) {
  const float2 x = upk2(a), y = upk2(b);
  return pk2(__fmul_rn(x.x, y.x), __fmul_rn(x.y, y.y));
}
__device__ __forceinline__ u64 fma2(u64 a, u64 b, u64 c) {
  const float2 x = upk2(a), y = upk2(b), z = upk2(c);
  return pk2(__fmaf_rn(x.x, y.x, z.x), __fmaf_rn(x.y, y.y, z.y));
}
#endif

// ---- shared memory, mbarriers, TMA -------------------------------------------
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
// Bounded wait: false after kWaitLimit unsuccessful polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (unsigned i = 0; i < kWaitLimit; ++i)
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

// ---- element conversion --------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int kBytes = 4;
  static __device__ __forceinline__ float get(const float* p, int i) { return p[i]; }
  // P consecutive fp32 pairs (2P elements) starting at a 16-byte aligned element
  template <int P>
  static __device__ __forceinline__ void pairs(const float* p, u64 (&out)[P]) {
    if constexpr (P % 2 == 0) {
#pragma unroll
      for (int k = 0; k < P / 2; ++k) {
        const ulonglong2 v = reinterpret_cast<const ulonglong2*>(p)[k];
        out[2 * k] = v.x;
        out[2 * k + 1] = v.y;
      }
    } else {
#pragma unroll
      for (int k = 0; k < P; ++k) out[k] = reinterpret_cast<const u64*>(p)[k];
    }
  }
  static __device__ __forceinline__ void put(float* p, int64_t i, float v) { p[i] = v; }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  static __device__ __forceinline__ float get(const __nv_bfloat16* p, int i) {
    return __bfloat162float(p[i]);
  }
  static __device__ __forceinline__ u64 widen(uint32_t w) {  // bf16x2 -> fp32 pair, exact
    return pk2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  template <int P>
  static __device__ __forceinline__ void pairs(const __nv_bfloat16* p, u64 (&out)[P]) {
    if constexpr (P % 4 == 0) {
#pragma unroll
      for (int k = 0; k < P / 4; ++k) {
        const uint4 v = reinterpret_cast<const uint4*>(p)[k];
        out[4 * k] = widen(v.x);
        out[4 * k + 1] = widen(v.y);
        out[4 * k + 2] = widen(v.z);
        out[4 * k + 3] = widen(v.w);
      }
    } else if constexpr (P % 2 == 0) {
#pragma unroll
      for (int k = 0; k < P / 2; ++k) {
        const uint2 v = reinterpret_cast<const uint2*>(p)[k];
        out[2 * k] = widen(v.x);
        out[2 * k + 1] = widen(v.y);
      }
    } else {
#pragma unroll
      for (int k = 0; k < P; ++k) out[k] = widen(reinterpret_cast<const uint32_t*>(p)[k]);
    }
  }
  static __device__ __forceinline__ void put(__nv_bfloat16* p, int64_t i, float v) {
    p[i] = __float2bfloat16_rn(v);
  }
};

// Sum over the NG lanes of a channel, scattered: lane g of the channel returns
// the full sum for step g of the NG partials it was given.  Each round halves
// the values a lane holds: it keeps the half selected by its lane bit and adds
// the half its partner sends (shuffles, so the shared-memory pipe stays free
// for the input loads).
template <int NG>
__device__ __forceinline__ float reduce_scatter(float (&v)[NG], int g) {
#pragma unroll
  for (int m = NG / 2; m >= 1; m /= 2) {
    const bool upper = (g & m) != 0;
#pragma unroll
    for (int k = 0; k < m; ++k) {
      const float keep = upper ? v[k + m] : v[k];
      const float send = upper ? v[k] : v[k + m];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
  }
  return v[0];
}

template <int N_, int NG_, int T_, int STAGES_, int WPC_, typename IO_, bool GATE_, int TS_ = 1>
struct Cfg {
  static constexpr int N = N_, NG = NG_, T = T_, STAGES = STAGES_, WPC = WPC_, TS = TS_;
  static constexpr bool GATE = GATE_;
  using IO = IO_;
  static constexpr int G = N / NG;          // states per lane
  static constexpr int P = G / 2;           // state pairs per lane
  static constexpr int CH = 32 / NG / TS;   // channels per warp
  // time split (TS = 2): each half-warp takes KS consecutive steps of a
  // sub-tile of TS * KS steps
  static constexpr int KS = 8;
  static constexpr int SUB = TS * KS;
  static constexpr int CPC = CH * WPC;      // channels per CTA
  // Steps per input batch: about 8 state pairs of inputs formed ahead.
  static constexpr int U = (8 / P < 1) ? 1 : (8 / P > NG ? NG : 8 / P);
  static constexpr int NB = NG / U;                      // batches per reduce group
  static constexpr int BODY = NB < 2 ? 2 : NB;           // batches per pipelined body
  static constexpr int BODY_STEPS = BODY * U;
  static constexpr int PAD = U;             // rows read past a tile by the last prefetch
  static constexpr int ES = Elem<IO>::kBytes;
  // stage slot: x, delta (, z) tiles [T + PAD][CPC]; B, C tiles [T + PAD][N]
  static constexpr int ACT = ((T + PAD) * CPC * ES + 127) / 128 * 128;
  static constexpr int ROW = ((T + PAD) * N * ES + 127) / 128 * 128;
  static constexpr int STAGE_BYTES = ACT * (GATE ? 3 : 2) + 2 * ROW;
  static constexpr int TX_BYTES = T * CPC * ES * (GATE ? 3 : 2) + 2 * T * N * ES;
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int SMEM = BAR_OFF + 2 * STAGES * 8;
  static_assert(G >= 2 && G % 2 == 0, "a lane holds whole state pairs");
  static_assert(NG >= 2 && NG <= 8 && (NG & (NG - 1)) == 0, "NG is 2, 4 or 8");
  static_assert((CPC * ES) % 16 == 0 && (N * ES) % 16 == 0, "TMA box rows are 16-byte multiples");
  static_assert(T <= 256 && T % NG == 0 && T % BODY_STEPS == 0, "tile steps");
  static_assert(NG % U == 0 && BODY % 2 == 0, "pipelined body alternates two input buffers");
  static_assert(TS == 1 || (TS == 2 && KS % NG == 0 && T % SUB == 0), "time split shape");
};

template <class K>
struct Slot {
  using IO = typename K::IO;
  __device__ static IO* x(char* s) { return reinterpret_cast<IO*>(s); }
  __device__ static IO* dt(char* s) { return reinterpret_cast<IO*>(s + K::ACT); }
  __device__ static IO* z(char* s) { return reinterpret_cast<IO*>(s + 2 * K::ACT); }
  __device__ static IO* B(char* s) { return reinterpret_cast<IO*>(s + K::ACT * (K::GATE ? 3 : 2)); }
  __device__ static IO* C(char* s) {
    return reinterpret_cast<IO*>(s + K::ACT * (K::GATE ? 3 : 2) + K::ROW);
  }
};

// Issue the TMA copies of one tile into a slot (one thread).
template <class K>
__device__ __forceinline__ void load_tile(char* slot, uint64_t* full, const CUtensorMap* tx,
                                          const CUtensorMap* tdt, const CUtensorMap* tz,
                                          const CUtensorMap* tb, const CUtensorMap* tc, int d0,
                                          int t0, int b) {
  mbar_expect_tx(full, K::TX_BYTES);
  tma_load_3d(Slot<K>::x(slot), tx, d0, t0, b, full);
  tma_load_3d(Slot<K>::dt(slot), tdt, d0, t0, b, full);
  if (K::GATE) tma_load_3d(Slot<K>::z(slot), tz, d0, t0, b, full);
  tma_load_3d(Slot<K>::B(slot), tb, 0, t0, b, full);
  tma_load_3d(Slot<K>::C(slot), tc, 0, t0, b, full);
}

// Inputs of one step for this lane's states: Abar = exp(delta A) as
// 2^(delta * A log2 e) ([P1] s2.4), the input term delta * B * x ([P1] s3.3),
// the C row and x.  `dl` / `xl` point at this lane's channel in the delta and
// x tiles (row stride CPC), `brow` / `crow` at this lane's slice of the B and
// C rows of the step.
template <class K>
__device__ __forceinline__ void step_inputs(const typename K::IO* dl, const typename K::IO* xl,
                                            const typename K::IO* brow, const typename K::IO* crow,
                                            const u64 (&a2)[K::P], u64 (&ab)[K::P],
                                            u64 (&bi)[K::P], u64 (&cq)[K::P], float& xv) {
  using E = Elem<typename K::IO>;
  const float dt = E::get(dl, 0);
  xv = E::get(xl, 0);
  const float uu = dt * xv;
  const u64 dd = pk2(dt, dt), ux = pk2(uu, uu);
  u64 bq[K::P];
  E::template pairs<K::P>(brow, bq);
  E::template pairs<K::P>(crow, cq);
#pragma unroll
  for (int q = 0; q < K::P; ++q) {
    const float2 arg = upk2(mul2(a2[q], dd));
    ab[q] = pk2(ex2(arg.x), ex2(arg.y));
    bi[q] = mul2(bq[q], ux);
  }
}

// As step_inputs, without the C row (the first pass of a time-split run).
template <class K>
__device__ __forceinline__ void step_inputs_ab(const typename K::IO* dl, const typename K::IO* xl,
                                               const typename K::IO* brow, const u64 (&a2)[K::P],
                                               u64 (&ab)[K::P], u64 (&bi)[K::P], float& xv) {
  using E = Elem<typename K::IO>;
  const float dt = E::get(dl, 0);
  xv = E::get(xl, 0);
  const float uu = dt * xv;
  const u64 dd = pk2(dt, dt), ux = pk2(uu, uu);
  u64 bq[K::P];
  E::template pairs<K::P>(brow, bq);
#pragma unroll
  for (int q = 0; q < K::P; ++q) {
    const float2 arg = upk2(mul2(a2[q], dd));
    ab[q] = pk2(ex2(arg.x), ex2(arg.y));
    bi[q] = mul2(bq[q], ux);
  }
}

// One step of h = Abar h + delta B x for this lane's states ([P1] s1.1), and
// this lane's part of the output sum_n C_n h_n (+ D x on the channel's lane 0,
// so the reduction over the channel's lanes also adds the D residual).
template <class K>
__device__ __forceinline__ float step_update(u64 (&h2)[K::P], const u64 (&ab)[K::P],
                                             const u64 (&bi)[K::P], const u64 (&cq)[K::P],
                                             float xv, float dg) {
  u64 acc = 0;
#pragma unroll
  for (int q = 0; q < K::P; ++q) {
    h2[q] = fma2(ab[q], h2[q], bi[q]);
    acc = q == 0 ? mul2(cq[q], h2[q]) : fma2(cq[q], h2[q], acc);
  }
  const float2 a = upk2(acc);
  return fmaf(dg, xv, a.x + a.y);
}

// The inputs of U consecutive steps, formed ahead of the recurrence.
template <class K>
struct Batch {
  u64 ab[K::U][K::P], bi[K::U][K::P], cq[K::U][K::P];
  float xv[K::U];
};

template <class K>
__device__ __forceinline__ void batch_inputs(const typename K::IO* dl, const typename K::IO* xl,
                                             const typename K::IO* brow,
                                             const typename K::IO* crow, int s,
                                             const u64 (&a2)[K::P], Batch<K>& bt) {
#pragma unroll
  for (int u = 0; u < K::U; ++u)
    step_inputs<K>(dl + (s + u) * K::CPC, xl + (s + u) * K::CPC, brow + (s + u) * K::N,
                   crow + (s + u) * K::N, a2, bt.ab[u], bt.bi[u], bt.cq[u], bt.xv[u]);
}

template <class K>
__device__ __forceinline__ void batch_update(u64 (&h2)[K::P], const Batch<K>& bt, float dg,
                                             float (&part)[K::BODY_STEPS], int off) {
#pragma unroll
  for (int u = 0; u < K::U; ++u)
    part[off + u] = step_update<K>(h2, bt.ab[u], bt.bi[u], bt.cq[u], bt.xv[u], dg);
}

template <class K>
__global__ void __launch_bounds__(K::WPC * 32)
    stream_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dt,
                  const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_b,
                  const __grid_constant__ CUtensorMap tm_c, const ScanParams p) {
  using IO = typename K::IO;
  using E = Elem<IO>;
  // Dynamic shared memory: the stage ring, then the
  // mbarriers.  Used through pointers derived from the __shared__ array so
  // that every access compiles to a shared-memory instruction.
  extern __shared__ __align__(128) char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + K::BAR_OFF);
  uint64_t* empty = full + K::STAGES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int64_t n_cg = (p.dim + K::CPC - 1) / K::CPC;
  const int64_t b = blockIdx.x / n_cg;
  const int d0 = static_cast<int>((blockIdx.x % n_cg) * K::CPC);
  const int hf = K::TS == 2 ? lane >> 4 : 0;      // time half of this lane (TS = 2)
  const int cw = (lane % (32 / K::TS)) / K::NG;    // channel within the warp
  const int c_loc = warp * K::CH + cw;             // channel within the CTA tile
  const int g = lane % K::NG;                      // state group of this lane
  const int64_t d = d0 + c_loc;
  const bool d_ok = d < p.dim;
  const int64_t L = p.seqlen;
  const int64_t lv = valid_steps(p, b);
  const int n_tiles = static_cast<int>((lv + K::T - 1) / K::T);  // tiles with a valid step
  const bool producer = threadIdx.x == 0;

  if (producer) {
    for (int st = 0; st < K::STAGES; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], K::WPC);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (producer) {
    for (int st = 0; st < K::STAGES && st < n_tiles; ++st)
      load_tile<K>(smem + st * K::STAGE_BYTES, &full[st], &tm_x, &tm_dt, &tm_z, &tm_b, &tm_c, d0,
                   st * K::T, static_cast<int>(b));
  }

  // per-lane constants: log2(e)-scaled A of this lane's states, D residual
  u64 a2[K::P], h2[K::P];
#pragma unroll
  for (int q = 0; q < K::P; ++q) {
    float lo = 0.f, hi = 0.f;
    if (d_ok) {
      lo = __ldg(p.A + d * K::N + g * K::G + 2 * q) * kLog2e;
      hi = __ldg(p.A + d * K::N + g * K::G + 2 * q + 1) * kLog2e;
    }
    a2[q] = pk2(lo, hi);
    h2[q] = pk2(0.f, 0.f);  // [P1] s4.1: h_0 = 0 unless given
    if (d_ok && p.h0)
      h2[q] = *reinterpret_cast<const u64*>(p.h0 + (b * p.dim + d) * K::N + g * K::G + 2 * q);
  }
  const float dskip = (d_ok && p.D) ? __ldg(p.D + d) : 0.f;
  const float dg = g == 0 ? dskip : 0.f;  // the channel's lane 0 adds D x to its partial
  IO* __restrict__ yout = static_cast<IO*>(p.y);
  const bool want_states = p.states != nullptr;
  // Chunk c ends at step min((c+1) chunk_len, L) - 1 ([P1] s3.4).
  auto chunk_end = [&](int64_t c) { return min((c + 1) * p.chunk_len, L) - 1; };
  int64_t next_c = 0;                                          // next chunk to store
  int64_t next_ce = want_states ? chunk_end(0) : INT64_MAX;    // its last step

  auto store_state = [&](int64_t t) {
    if (d_ok) {
      float* sp = p.states + ((b * p.n_chunks + t / p.chunk_len) * p.dim + d) * K::N + g * K::G;
#pragma unroll
      for (int q = 0; q < K::P; ++q) reinterpret_cast<float2*>(sp)[q] = upk2(h2[q]);
    }
  };

  bool ok = true;
  for (int i = 0; i < n_tiles && ok; ++i) {
    const int slot = i % K::STAGES;
    char* st = smem + slot * K::STAGE_BYTES;
    ok = mbar_wait(&full[slot], (i / K::STAGES) & 1);
    if (!ok) break;
    // refill the slot freed by the previous tile (all warps are done with it)
    if (producer && i >= 1 && i - 1 + K::STAGES < n_tiles) {
      const int ps = (i - 1) % K::STAGES;
      ok = mbar_wait(&empty[ps], ((i - 1) / K::STAGES) & 1);
      if (ok)
        load_tile<K>(smem + ps * K::STAGE_BYTES, &full[ps], &tm_x, &tm_dt, &tm_z, &tm_b, &tm_c,
                     d0, (i - 1 + K::STAGES) * K::T, static_cast<int>(b));
    }
    const IO* xs = Slot<K>::x(st);
    const IO* zs = Slot<K>::z(st);
    const int64_t t0 = static_cast<int64_t>(i) * K::T;
    const int steps = static_cast<int>(lv - t0 < K::T ? lv - t0 : K::T);  // valid steps in tile

    const IO* dl = Slot<K>::dt(st) + c_loc;                          // this lane's channel
    const IO* xl = xs + c_loc;
    const IO* b_l = Slot<K>::B(st) + g * K::G;                        // this lane's states
    const IO* c_l = Slot<K>::C(st) + g * K::G;
    IO* yrow = yout + (b * L + t0) * p.dim + d;                       // y[b, t0, d]

    // Output of one finished group [s, s + NG): a shuffle reduce-scatter over
    // the channel's NG lanes leaves lane g with the full sum of step s + g
    // (sum_n C_n h_n + D x); the gate and the store follow.
    auto finish_group = [&](float (&v)[K::NG], int s) {
      float yv = reduce_scatter<K::NG>(v, g);
      const int sg = s + g;
      if (d_ok && sg < steps) {
        if (K::GATE) yv *= silu(E::get(zs, sg * K::CPC + c_loc));  // * silu(z)
        E::put(yrow, static_cast<int64_t>(sg) * p.dim, yv);
      }
    };

    if constexpr (K::TS == 2) {
      // Time split: half-warp hf takes steps [s + hf KS, s + hf KS + KS) of each
      // sub-tile.  Each lane folds its run into (A, Bsum) keeping every step's
      // (a, b) ([P1] s3.1 first level), the halves exchange the state in one
      // shuffle round (a two-element Hillis-Steele scan, [P1] s2.2), and both
      // replay their runs to form h and C h.
      for (int s = 0; s < steps; s += K::SUB) {
        const int r0 = s + hf * K::KS;                        // first step of this lane's run
        const int64_t sub_end = t0 + s + K::SUB - 1;          // last step of the sub-tile
        const bool full = s + K::SUB <= steps;
        const bool inner_ce = next_ce < sub_end;              // a chunk end before the last step
        u64 ab[K::KS][K::P], bi[K::KS][K::P];
        float xv[K::KS];
#pragma unroll
        for (int j = 0; j < K::KS; ++j) {
          step_inputs_ab<K>(dl + (r0 + j) * K::CPC, xl + (r0 + j) * K::CPC, b_l + (r0 + j) * K::N,
                            a2, ab[j], bi[j], xv[j]);
          if (!full && r0 + j >= steps) {  // identity step (a = 1, b = 0), [P1] s2.3
#pragma unroll
            for (int q = 0; q < K::P; ++q) { ab[j][q] = pk2(1.f, 1.f); bi[j][q] = pk2(0.f, 0.f); }
          }
        }
        u64 A[K::P], Bs[K::P], h[K::P];
#pragma unroll
        for (int q = 0; q < K::P; ++q) {
          A[q] = ab[0][q];
          Bs[q] = bi[0][q];
#pragma unroll
          for (int j = 1; j < K::KS; ++j) {  // (A, Bs) o (a_j, b_j)
            Bs[q] = fma2(ab[j][q], Bs[q], bi[j][q]);
            A[q] = mul2(A[q], ab[j][q]);
          }
          // state after the first half, sent to the second half
          const float2 e1 = upk2(fma2(A[q], h2[q], Bs[q]));
          const float r1x = __shfl_xor_sync(0xffffffffu, e1.x, 16);
          const float r1y = __shfl_xor_sync(0xffffffffu, e1.y, 16);
          h[q] = hf ? pk2(r1x, r1y) : h2[q];                  // state before this lane's run
          const float2 e2 = upk2(fma2(A[q], h[q], Bs[q]));    // second half: sub-tile end
          const float r2x = __shfl_xor_sync(0xffffffffu, e2.x, 16);
          const float r2y = __shfl_xor_sync(0xffffffffu, e2.y, 16);
          h2[q] = hf ? pk2(e2.x, e2.y) : pk2(r2x, r2y);       // carried to the next sub-tile
        }
        float part[K::KS];
        int64_t ce = INT64_MAX;  // first chunk end at or after this lane's run
        if (inner_ce) {
          ce = ((t0 + r0) / p.chunk_len + 1) * p.chunk_len - 1;
          if (ce > L - 1) ce = L - 1;
        }
#pragma unroll
        for (int j = 0; j < K::KS; ++j) {
          u64 cq[K::P];
          E::template pairs<K::P>(c_l + (r0 + j) * K::N, cq);
          u64 acc = 0;
#pragma unroll
          for (int q = 0; q < K::P; ++q) {
            h[q] = fma2(ab[j][q], h[q], bi[j][q]);
            acc = q == 0 ? mul2(cq[q], h[q]) : fma2(cq[q], h[q], acc);
          }
          const float2 a = upk2(acc);
          part[j] = fmaf(dg, xv[j], a.x + a.y);
          if (inner_ce && t0 + r0 + j == ce) {  // [P1] s3.4: a chunk ends inside this run
            if (d_ok) {
              float* sp = p.states + ((b * p.n_chunks + ce / p.chunk_len) * p.dim + d) * K::N +
                          g * K::G;
#pragma unroll
              for (int q = 0; q < K::P; ++q) reinterpret_cast<float2*>(sp)[q] = upk2(h[q]);
            }
            ce = ce + p.chunk_len > L - 1 ? (ce == L - 1 ? INT64_MAX : L - 1) : ce + p.chunk_len;
          }
        }
        // chunk ends in this sub-tile: interior ones were stored above by the
        // owning half; the one at the sub-tile's last step is the carried state
        while (next_ce <= sub_end) {
          if (next_ce == sub_end && hf == 1) store_state(next_ce);
          ++next_c;
          next_ce = next_c < p.n_chunks ? chunk_end(next_c) : INT64_MAX;
        }
#pragma unroll
        for (int k0 = 0; k0 < K::KS; k0 += K::NG) {
          float v[K::NG];
#pragma unroll
          for (int i2 = 0; i2 < K::NG; ++i2) v[i2] = part[k0 + i2];
          finish_group(v, r0 + k0);
        }
      }
    } else {
    int s0 = 0;
    while (s0 < steps) {
      // Longest run [s0, run_end) of whole bodies with no chunk end inside.
      int run_end = s0 + (steps - s0) / K::BODY_STEPS * K::BODY_STEPS;
      if (next_ce < t0 + run_end)
        run_end = s0 + static_cast<int>((next_ce - t0 - s0) / K::BODY_STEPS) * K::BODY_STEPS;
      if (run_end > s0) {
        // Software pipeline over batches of U steps: the inputs of the next
        // batch (loads, exps, delta*B*x) are formed while the current batch
        // runs its recurrence and finished groups are reduced.  The last
        // prefetch of a run reads at most PAD rows past it, inside the slot.
        Batch<K> bA, bB;
        batch_inputs<K>(dl, xl, b_l, c_l, s0, a2, bA);
        for (int s = s0; s < run_end; s += K::BODY_STEPS) {
          float part[K::BODY_STEPS];
#pragma unroll
          for (int k = 0; k < K::BODY; ++k) {
            const int sn = s + (k + 1) * K::U;
            if (k % 2 == 0) {
              batch_inputs<K>(dl, xl, b_l, c_l, sn, a2, bB);
              batch_update<K>(h2, bA, dg, part, k * K::U);
            } else {
              batch_inputs<K>(dl, xl, b_l, c_l, sn, a2, bA);
              batch_update<K>(h2, bB, dg, part, k * K::U);
            }
            if (((k + 1) * K::U) % K::NG == 0) {
              const int j = ((k + 1) * K::U) / K::NG - 1;  // group within the body
              float v[K::NG];
#pragma unroll
              for (int i2 = 0; i2 < K::NG; ++i2) v[i2] = part[j * K::NG + i2];
              finish_group(v, s + j * K::NG);
            }
          }
        }
        s0 = run_end;
      }
      if (s0 < steps) {
        // One group that holds a chunk end or runs past the last valid step.
        float part[K::NG];
#pragma unroll
        for (int u = 0; u < K::NG; ++u) {
          const int s = s0 + u;
          u64 ab[K::P], bi[K::P], cq[K::P];
          float xv;
          step_inputs<K>(dl + s * K::CPC, xl + s * K::CPC, b_l + s * K::N, c_l + s * K::N, a2,
                         ab, bi, cq, xv);
          if (s >= steps) {  // identity step (a = 1, b = 0), [P1] s2.3
#pragma unroll
            for (int q = 0; q < K::P; ++q) { ab[q] = pk2(1.f, 1.f); bi[q] = pk2(0.f, 0.f); }
          }
          part[u] = step_update<K>(h2, ab, bi, cq, xv, dg);
          if (t0 + s == next_ce) {  // [P1] s3.4 chunk boundary state
            store_state(next_ce);
            ++next_c;
            next_ce = next_c < p.n_chunks ? chunk_end(next_c) : INT64_MAX;
          }
        }
        finish_group(part, s0);
        s0 += K::NG;
      }
    }
    }  // TS
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
  if (!ok) {
    if (lane == 0) atomicOr(&g_stream_error, kErrWait);
    return;
  }

  // Steps past valid_len: exact zeros, frozen state for the remaining chunk ends.
  if (lv < L) {
    const int per = 32 / K::CH;  // steps covered by one pass of the warp
    const int cz = lane % K::CH, sz = lane / K::CH;  // (channel, step) of this lane
    const int64_t dz = d0 + warp * K::CH + cz;
    if (dz < p.dim)
      for (int64_t t = lv + sz; t < L; t += per) E::put(yout, (b * L + t) * p.dim + dz, 0.f);
  }
  if (want_states)
    for (; next_c < p.n_chunks; ++next_c) store_state(chunk_end(next_c));  // frozen state
  if (p.h_final && d_ok && hf == 0) {  // state after the last step
    float* fp = p.h_final + (b * p.dim + d) * K::N + g * K::G;
#pragma unroll
    for (int q = 0; q < K::P; ++q) reinterpret_cast<float2*>(fp)[q] = upk2(h2[q]);
  }
}

// ---- host side --------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

// 3-D map over a [batch, seqlen, inner] tensor with a box of {box_inner, box_t, 1}.
bool make_map(CUtensorMap* m, const void* base, bool bf16, int64_t inner, int64_t L, int64_t batch,
              int box_inner, int box_t) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || base == nullptr) return false;
  const int es = bf16 ? 2 : 4;
  cuuint64_t dims[3] = {cuuint64_t(inner), cuuint64_t(L), cuuint64_t(batch)};
  cuuint64_t strides[2] = {cuuint64_t(inner * es), cuuint64_t(inner * L * es)};
  cuuint32_t box[3] = {cuuint32_t(box_inner), cuuint32_t(box_t), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <class K>
cudaError_t launch_k(const ScanParams& p, cudaStream_t s) {
  const bool bf16 = sizeof(typename K::IO) == 2;
  CUtensorMap mx, mdt, mz, mb, mc;
  if (!make_map(&mx, p.x, bf16, p.dim, p.seqlen, p.batch, K::CPC, K::T) ||
      !make_map(&mdt, p.delta, bf16, p.dim, p.seqlen, p.batch, K::CPC, K::T) ||
      !make_map(&mb, p.B, bf16, K::N, p.seqlen, p.batch, K::N, K::T) ||
      !make_map(&mc, p.C, bf16, K::N, p.seqlen, p.batch, K::N, K::T))
    return cudaErrorInvalidValue;
  if (K::GATE) {
    if (!make_map(&mz, p.z, bf16, p.dim, p.seqlen, p.batch, K::CPC, K::T))
      return cudaErrorInvalidValue;
  } else {
    mz = mx;  // unused
  }
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(stream_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         K::SMEM);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int64_t n_cg = (p.dim + K::CPC - 1) / K::CPC;
  const int64_t grid = n_cg * p.batch;
  stream_kernel<K><<<static_cast<unsigned>(grid), K::WPC * 32, K::SMEM, s>>>(mx, mdt, mz, mb, mc, p);
  return cudaGetLastError();
}

// Tile length (steps per TMA copy) and ring depth; overridable at build time.
#ifndef SSM_STREAM_T
#define SSM_STREAM_T 32
#endif
#ifndef SSM_STREAM_STAGES
#define SSM_STREAM_STAGES 4
#endif

// Instances: (N, NG = N / G) per state size, tile T, ring depth, warps per CTA.
#define SSM_STREAM_INSTANCES(X)                                          \
  X(8, 4, 1, 1) X(8, 4, 2, 1)                                            \
  X(16, 4, 1, 1) X(16, 4, 2, 1) X(16, 4, 4, 1) X(16, 8, 2, 1)            \
  X(16, 4, 2, 2) X(16, 4, 4, 2)                                          \
  X(32, 4, 2, 1) X(32, 8, 2, 1) X(32, 4, 4, 2)                           \
  X(64, 8, 2, 1) X(64, 8, 4, 1) X(64, 16, 2, 1) X(64, 8, 4, 2)

template <typename IO, bool GATE>
cudaError_t launch_io(const ScanParams& p, cudaStream_t s, StreamShape sh) {
#define SSM_CASE(n_, g_, w_, ts_)                                                     \
  if (p.dstate == n_ && sh.g == g_ && sh.wpc == w_ && sh.ts == ts_)                   \
    return launch_k<Cfg<n_, n_ / g_, SSM_STREAM_T, SSM_STREAM_STAGES, w_, IO, GATE, ts_>>(p, s);
  SSM_STREAM_INSTANCES(SSM_CASE)
#undef SSM_CASE
  return cudaErrorInvalidValue;
}

bool has_instance(int n, int g, int w, int ts) {
#define SSM_HAS(n_, g_, w_, ts_) if (n == n_ && g == g_ && w == w_ && ts == ts_) return true;
  SSM_STREAM_INSTANCES(SSM_HAS)
#undef SSM_HAS
  return false;
}

}  // namespace

StreamShape stream_shape(const ScanParams& p, int warps_per_block, int states_per_lane,
                         int time_split) {
  StreamShape sh;
  sh.g = states_per_lane ? states_per_lane : (p.dstate >= 64 ? 8 : 4);
  sh.wpc = warps_per_block ? warps_per_block : 2;
  sh.ts = time_split ? time_split : 1;
  if (!has_instance(p.dstate, sh.g, sh.wpc, sh.ts)) return StreamShape{0, 0, 0};
  return sh;
}

static int stream_cpc(StreamShape sh, int dstate) {
  return sh.g ? (32 / (dstate / sh.g) / sh.ts) * sh.wpc : 0;
}

bool read_and_clear_device_errors(unsigned int* word) {
  unsigned int zero = 0;
  if (cudaMemcpyFromSymbol(word, g_stream_error, sizeof(unsigned int)) != cudaSuccess) return false;
  return cudaMemcpyToSymbol(g_stream_error, &zero, sizeof(unsigned int)) == cudaSuccess;
}

bool stream_eligible(const ScanParams& p, bool bf16, StreamShape sh) {
  const int es = bf16 ? 2 : 4;
  const int cpc = stream_cpc(sh, p.dstate);
  if (cpc == 0) return false;
  if (p.dstate * es < 16 || (cpc * es) % 16 != 0) return false;
  if ((p.dim * es) % 16 != 0) return false;
  if (p.seqlen > INT32_MAX || p.batch > INT32_MAX) return false;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(p.x) | reinterpret_cast<uintptr_t>(p.delta) |
                        reinterpret_cast<uintptr_t>(p.B) | reinterpret_cast<uintptr_t>(p.C) |
                        reinterpret_cast<uintptr_t>(p.z);
  if (mis % 16 != 0) return false;
  if ((reinterpret_cast<uintptr_t>(p.h0) | reinterpret_cast<uintptr_t>(p.h_final)) % 8 != 0)
    return false;
  if (encode_fn() == nullptr) return false;
  const int64_t grid = (p.dim + cpc - 1) / cpc * p.batch;
  return grid <= INT32_MAX;
}

int64_t stream_grid(const ScanParams& p, StreamShape sh) {
  const int cpc = stream_cpc(sh, p.dstate);
  return cpc ? (p.dim + cpc - 1) / cpc * p.batch : 0;
}

cudaError_t launch_stream(const ScanParams& p, bool bf16, cudaStream_t s, StreamShape sh) {
  if (bf16)
    return p.z ? launch_io<__nv_bfloat16, true>(p, s, sh) : launch_io<__nv_bfloat16, false>(p, s, sh);
  return p.z ? launch_io<float, true>(p, s, sh) : launch_io<float, false>(p, s, sh);
}

}  // namespace ssm
