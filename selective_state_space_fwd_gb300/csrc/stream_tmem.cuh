// stream_tmem.cuh -- STREAM-TM: the register sweep of the STREAM tier with the
// B and C rows delivered to every lane through tensor memory.
//
// Why.  In the STREAM tier every lane loads the B and C values of its states
// from shared memory at every step; 32 lanes reading the same few 16-byte
// chunks still cost the full 512 bytes of register delivery per load, and
// those loads are most of the kernel's shared-memory traffic (the unit that
// bounds it).  Here the rows are broadcast once per CTA into tensor memory
// (TMEM), whose loads into registers run several times faster than shared
// memory, and the lanes read them with tcgen05.ld.
//
// The broadcast is one tensor-core product per group of steps.  Lane l of a
// warp holds G consecutive states of one channel: state group sg(l) = l mod NG.
// The product D = S P, with S the 128 x K selection matrix (row m = TMEM lane
// m: 1 in the K entries of its lane's state group, else 0) and P the K x 256
// matrix whose column (step, j) holds, for every state group, the value B or C
// of that step and state split exactly into three bf16 pieces
// (v = hi + mid + lo, hi and mid truncations, lo the remainder), puts into
// TMEM lane m, column (step, j) the value of lane m's own state: products by
// 0 and 1 are exact and the three pieces sum back to v exactly in the fp32
// accumulator whenever the low piece is a normal number (|v| >= 2^-109; below,
// its last bits are lost: relative error under 2^-15, absolute under 2^-125).
// Columns per batch of U steps (U G = 8): the 8 values of B, then the 8 of C.
//
// Arithmetic per lane and step: one channel x G states as G/2 f32x2 pairs
// over consecutive STATES (the B, C pairs come straight from the TMEM
// registers; delta and delta*x are duplicated into pairs once per step).  Per
// (channel, state): one MUFU ex2 and four fp32 operations, as in STREAM
// ([P1] s2.4 Abar = exp(delta A), s3.3 b = delta B x, the update, the C
// contraction).  The C contraction over the NG lanes of a channel goes through
// a per-warp shared buffer and a block epilogue that adds D x, applies the
// silu(z) gate and stores y ([P1] s3.3: h never leaves registers).
//
// CTA: W compute warps (TMEM lane quadrant w mod 4; every quadrant holds the
// same broadcast) plus one producer warp that issues the TMA copies of the
// x, delta (, z) slabs and B, C rows, builds the product operands and issues
// the products.  TMEM holds two groups of 256 columns (double buffer).  Every
// mbarrier wait is bounded: a wait that gives up sets the sticky error word
// and an abort flag that stops the other warps; before the CTA exits, the
// producer waits (bounded) for its products and copies in flight and frees
// the TMEM it holds.
#pragma once

#include <cuda.h>

#include "stream_core.cuh"
#include "umma.cuh"

namespace ssm {
namespace stream_tm {

using stream::fma2;
using stream::mul2;
using stream::pk2;
using stream::u64;
using stream::upk2;

constexpr unsigned kErrWaitTm = 8u;  // sticky error bit of this tier's bounded waits

template <int N_, int G_, int R_, int W_, typename IO_, bool GATE_>
struct Cfg {
  static constexpr int N = N_, G = G_, R = R_, W = W_;
  using IO = IO_;
  static constexpr bool GATE = GATE_;
  static constexpr int NG = N / G;            // lanes (state groups) per channel
  static constexpr int CW = 32 / NG * R;      // channels per warp
  static constexpr int GP = G / 2;            // state pairs per lane
  static constexpr int T = 64;                // steps per TMA tile
  static constexpr int M = 16;                // steps per epilogue block
  static constexpr int SPG = 128 / G;         // steps per TMEM group (2G columns per step, 256 per group)
  static constexpr int U = G <= 4 ? 2 : 1;    // steps per load batch (16 TMEM columns)
  static constexpr int BCOLS = U * 2 * G;     // TMEM columns of one batch
  static constexpr int KS = (3 * NG + 15) / 16;  // K-steps of 16 of the broadcast product
  static constexpr int ES = stream::Tile<IO>::kBytes;
  static constexpr int SLAB = T * CW * ES;    // one warp's [T x CW] tile of one tensor
  static constexpr int ROWT = T * N * ES;     // [T x N] tile of B or C
  static constexpr int NACT = GATE ? 3 : 2;
  static constexpr int STAGE = NACT * W * SLAB + 2 * ROWT;
  static constexpr int PS = stream::pad_ps(NG, CW, R);
  static constexpr int PROW = stream::pad_prow(NG, CW, R, PS);
  static constexpr int PBYTES = M * PROW * 4;
  // The product operands (bf16, core matrices of 8 rows x 16 bytes).  S is
  // K-major (core matrices 128 bytes apart along K, 256 along M).  P is
  // MN-major: a core matrix holds 8 K-rows of 8 consecutive columns; K-groups
  // are 128 bytes apart and 8-column groups OSBO bytes apart, a stride chosen
  // so that the producer's 16-byte stores of one access phase hit distinct
  // banks.
  static constexpr int OSBO = 320;
  static constexpr int OBYTES = 32 * OSBO;    // one K-step of P: 256 columns x 16 K
  static constexpr int ABYTES = 128 * 16 * 2; // one K-step of S: 128 rows x 16 K
  // TMEM columns of a batch of U steps: the U x G values of B (step-major),
  // then those of C; both halves are 8 columns (one 16-byte MN-major row of
  // the operand).  Producer items: (batch, state group), 16 columns each.
  static constexpr int ITEMS = SPG / U * NG;  // per group
  static_assert(U * G == 8, "a batch holds 8 values of B and 8 of C per lane");
  static_assert(ITEMS % 32 == 0, "producer items");
  static constexpr int TCOLS = 512;           // two groups of 256 columns
  static_assert(G == 4 || G == 8, "four or eight states per lane");
  static_assert(N % G == 0 && NG >= 1 && NG <= 8, "state groups");
  static_assert((CW * ES) % 16 == 0 && (N * ES) % 16 == 0, "TMA box rows are 16-byte multiples");
  static_assert(T % SPG == 0 && SPG % M == 0 && M % (2 * U) == 0 && M % NG == 0, "steps");
  static_assert(SLAB % 128 == 0 && ROWT % 128 == 0, "slot alignment");
  static_assert(W == 4 || W == 8, "compute warps per CTA");
  static_assert(R == 1 || R == 2, "one channel or a pair of channels per lane");
};

struct LaunchArgs {
  int stages;
  unsigned int* err;
};

// ---- tensor memory loads of one batch (U steps x 2G columns) ------------------
template <int NC>
struct TReg {
  uint32_t r[NC];
};
__device__ __forceinline__ void tld(uint32_t taddr, TReg<16>& v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v.r[0]), "=r"(v.r[1]), "=r"(v.r[2]), "=r"(v.r[3]), "=r"(v.r[4]), "=r"(v.r[5]),
        "=r"(v.r[6]), "=r"(v.r[7]), "=r"(v.r[8]), "=r"(v.r[9]), "=r"(v.r[10]), "=r"(v.r[11]),
        "=r"(v.r[12]), "=r"(v.r[13]), "=r"(v.r[14]), "=r"(v.r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tld(uint32_t taddr, TReg<8>& v) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v.r[0]), "=r"(v.r[1]), "=r"(v.r[2]), "=r"(v.r[3]), "=r"(v.r[4]),
                 "=r"(v.r[5]), "=r"(v.r[6]), "=r"(v.r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tld_wait(TReg<8>& v) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v.r[0]), "+r"(v.r[1]), "+r"(v.r[2]), "+r"(v.r[3]), "+r"(v.r[4]),
                 "+r"(v.r[5]), "+r"(v.r[6]), "+r"(v.r[7])::"memory");
}
__device__ __forceinline__ void tld_wait(TReg<8>& v, TReg<8>& w) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v.r[0]), "+r"(v.r[1]), "+r"(v.r[2]), "+r"(v.r[3]), "+r"(v.r[4]),
                 "+r"(v.r[5]), "+r"(v.r[6]), "+r"(v.r[7]), "+r"(w.r[0]), "+r"(w.r[1]),
                 "+r"(w.r[2]), "+r"(w.r[3]), "+r"(w.r[4]), "+r"(w.r[5]), "+r"(w.r[6]),
                 "+r"(w.r[7])::"memory");
}
// Wait for this thread's outstanding TMEM loads; ties the batch registers to
// the wait so that no use of them moves above it.
__device__ __forceinline__ void tld_wait(TReg<16>& v) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v.r[0]), "+r"(v.r[1]), "+r"(v.r[2]), "+r"(v.r[3]), "+r"(v.r[4]),
                 "+r"(v.r[5]), "+r"(v.r[6]), "+r"(v.r[7]), "+r"(v.r[8]), "+r"(v.r[9]),
                 "+r"(v.r[10]), "+r"(v.r[11]), "+r"(v.r[12]), "+r"(v.r[13]), "+r"(v.r[14]),
                 "+r"(v.r[15])::"memory");
}

// ---- bounded waits that also stop when another warp gave up -------------------
__device__ __forceinline__ bool wait_tm(uint64_t* bar, uint32_t parity, volatile int* abort) {
  for (unsigned i = 0; i < stream::kWaitLimit; ++i) {
    if (stream::mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort) return false;
  }
  *abort = 1;
  return false;
}

// Three exact bf16 pieces of v (hi, mid: truncations; lo: the remainder), as
// bf16 bit patterns in the low 16 bits.
__device__ __forceinline__ void split3(float v, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
  const uint32_t vb = __float_as_uint(v);
  const float h = __uint_as_float(vb & 0xFFFF0000u);
  const float r = v - h;  // exact
  const uint32_t rb = __float_as_uint(r);
  const float m = __uint_as_float(rb & 0xFFFF0000u);
  const float l = r - m;  // exact
  hi = vb >> 16;
  mid = rb >> 16;
  lo = __float_as_uint(l) >> 16;
}

// The bf16 bit patterns in the upper halves of two fp32 words, packed
// (a in the low half).
__device__ __forceinline__ uint32_t hi_pair(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x7632); }

// Pieces of 8 values v[0..7] (8 consecutive operand columns of one K-row
// each): for piece p, 4 words of bf16 pairs.
__device__ __forceinline__ void split8(const float (&v)[8], uint4 (&out)[3]) {
  uint32_t h[8], m[8], l[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t vb = __float_as_uint(v[i]);
    const uint32_t hb = vb & 0xFFFF0000u;
    const float r = v[i] - __uint_as_float(hb);  // exact
    const uint32_t rb = __float_as_uint(r);
    const uint32_t mb = rb & 0xFFFF0000u;
    h[i] = vb;  // upper half = the truncated piece
    m[i] = rb;
    l[i] = __float_as_uint(r - __uint_as_float(mb));  // exact
  }
  out[0] = make_uint4(hi_pair(h[0], h[1]), hi_pair(h[2], h[3]), hi_pair(h[4], h[5]), hi_pair(h[6], h[7]));
  out[1] = make_uint4(hi_pair(m[0], m[1]), hi_pair(m[2], m[3]), hi_pair(m[4], m[5]), hi_pair(m[6], m[7]));
  out[2] = make_uint4(hi_pair(l[0], l[1]), hi_pair(l[2], l[3]), hi_pair(l[4], l[5]), hi_pair(l[6], l[7]));
}

// Eight consecutive stored elements widened to fp32 (16 or 32 bytes of shared memory).
template <typename IO>
__device__ __forceinline__ void load8(const IO* p, float (&v)[8]) {
  if constexpr (sizeof(IO) == 2) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(a[i] << 16);
      v[2 * i + 1] = __uint_as_float(a[i] & 0xFFFF0000u);
    }
  } else {
    const float4 x = *reinterpret_cast<const float4*>(p), y = *reinterpret_cast<const float4*>(p + 4);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
  }
}
template <typename IO>
__device__ __forceinline__ void load4(const IO* p, float* v) {
  if constexpr (sizeof(IO) == 2) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    v[0] = __uint_as_float(w.x << 16); v[1] = __uint_as_float(w.x & 0xFFFF0000u);
    v[2] = __uint_as_float(w.y << 16); v[3] = __uint_as_float(w.y & 0xFFFF0000u);
  } else {
    const float4 x = *reinterpret_cast<const float4*>(p);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  }
}

// Widen one stored element to fp32.
template <typename IO>
__device__ __forceinline__ float widen1(const IO* p) {
  if constexpr (sizeof(IO) == 2) return __uint_as_float(uint32_t(*reinterpret_cast<const uint16_t*>(p)) << 16);
  else return *reinterpret_cast<const float*>(p);
}

// Predicated store of one output element (bf16: round to nearest even).
template <typename IO>
__device__ __forceinline__ void put1(IO* p, float v, bool on) {
  if constexpr (sizeof(IO) == 2) {
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    const uint16_t w = *reinterpret_cast<const uint16_t*>(&b);
    asm volatile("{\n .reg .pred q;\n setp.ne.b32 q, %2, 0;\n @q st.global.b16 [%0], %1;\n}\n" ::"l"(p),
                 "h"(w), "r"(int(on)));
  } else {
    asm volatile("{\n .reg .pred q;\n setp.ne.b32 q, %2, 0;\n @q st.global.f32 [%0], %1;\n}\n" ::"l"(p),
                 "f"(v), "r"(int(on)));
  }
}

template <class K>
__global__ void __launch_bounds__((K::W + 1) * 32, 1)
    stream_tm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dt,
                     const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_b,
                     const __grid_constant__ CUtensorMap tm_c, const ScanParams p, const LaunchArgs la) {
  using IO = typename K::IO;
  constexpr int N = K::N, G = K::G, R = K::R, W = K::W, NG = K::NG, CW = K::CW, GP = K::GP;
  constexpr int T = K::T, M = K::M, U = K::U, SPG = K::SPG, KS = K::KS;
  extern __shared__ __align__(1024) char smem_raw[];
  // 1024-byte aligned base for the product operands
  char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int STAGES = la.stages;
  char* ring = smem;
  char* opA = ring + STAGES * K::STAGE;            // KS selection tiles
  char* opP = opA + KS * K::ABYTES;                // 2 groups x KS operand tiles
  float* pbufs = reinterpret_cast<float*>(opP + 2 * KS * K::OBYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<char*>(pbufs) + W * K::PBYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;   // [2]: a group's products are in TMEM
  uint64_t* tempty = tfull + 2;       // [2]: every compute warp is done reading a group
  uint32_t* tslot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cpc = W * CW;
  const int64_t n_cb = (p.dim + cpc - 1) / cpc;
  const int64_t b = blockIdx.x / n_cb;
  const int d0 = static_cast<int>((blockIdx.x % n_cb) * cpc);
  const int64_t L = p.seqlen;
  const int64_t lv = valid_steps(p, b);
  const int n_tiles = static_cast<int>((lv + T - 1) / T);
  // groups of a tile that hold a valid step
  auto tile_steps = [&](int i) { return static_cast<int>(lv - int64_t(i) * T < T ? lv - int64_t(i) * T : T); };
  auto tile_groups = [&](int i) { return (tile_steps(i) + SPG - 1) / SPG; };

  // ---- set-up: barriers, TMEM, the selection matrix ----------------------------
  if (warp == W) {
    if (lane == 0) {
      for (int s = 0; s < STAGES; ++s) {
        stream::mbar_init(&full[s], 1);
        stream::mbar_init(&empty[s], W);
      }
      for (int s = 0; s < 2; ++s) {
        stream::mbar_init(&tfull[s], 1);
        stream::mbar_init(&tempty[s], W);
      }
      *abort = 0;
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    umma::tmem_alloc(umma::smem_u32(tslot), K::TCOLS);
    // S: row m (TMEM lane m, lane m mod 32 of its warp) selects the three pieces
    // of its state group; K-major core matrices, 128 bytes apart along K, 256
    // bytes apart along M.
    for (int i = lane; i < KS * 128 * 8; i += 32) {  // pairs of K entries
      const int q = i / (128 * 8), rem = i % (128 * 8), m = rem / 8, kp = rem % 8;
      const int sg = (m & 31) % NG;
      uint32_t w = 0;
      for (int h = 0; h < 2; ++h) {
        const int k = q * 16 + kp * 2 + h;
        if (k < 3 * NG && k / 3 == sg) w |= 0x3F80u << (16 * h);  // bf16 1.0
      }
      const int kk = kp * 2;
      *reinterpret_cast<uint32_t*>(opA + q * K::ABYTES + (m >> 3) * 256 + (kk >> 3) * 128 +
                                   (m & 7) * 16 + (kk & 7) * 2) = w;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tbase = *tslot;

  if (warp == W) {
    // ================= producer warp ==============================================
    auto issue = [&](int tile, int slot) {
      char* st = ring + slot * K::STAGE;
      const int t0 = tile * T;
      stream::mbar_expect_tx(&full[slot], K::STAGE);
      for (int w = 0; w < W; ++w) {
        stream::tma_load_3d(st + (0 * W + w) * K::SLAB, &tm_x, d0 + w * CW, t0, int(b), &full[slot]);
        stream::tma_load_3d(st + (1 * W + w) * K::SLAB, &tm_dt, d0 + w * CW, t0, int(b), &full[slot]);
        if constexpr (K::GATE)
          stream::tma_load_3d(st + (2 * W + w) * K::SLAB, &tm_z, d0 + w * CW, t0, int(b), &full[slot]);
      }
      char* rows = st + K::NACT * W * K::SLAB;
      stream::tma_load_3d(rows, &tm_b, 0, t0, int(b), &full[slot]);
      stream::tma_load_3d(rows + K::ROWT, &tm_c, 0, t0, int(b), &full[slot]);
    };
    int issued = 0;  // tiles whose copies were issued
    if (lane == 0)
      for (; issued < STAGES && issued < n_tiles; ++issued) issue(issued, issued);
    issued = __shfl_sync(0xffffffffu, issued, 0);
    int waited = 0;  // tiles whose copies were waited for
    int g = 0;       // groups issued so far
    constexpr uint32_t idesc = umma::idesc_bf16(128, 256, false, true);
    bool ok = true;
    for (int i = 0; i < n_tiles && ok; ++i) {
      const int slot = i % STAGES;
      ok = wait_tm(&full[slot], (i / STAGES) & 1, abort);
      if (!ok) break;
      waited = i + 1;
      const int steps = tile_steps(i);
      const IO* rowB = reinterpret_cast<const IO*>(ring + slot * K::STAGE + K::NACT * W * K::SLAB);
      const IO* rowC = rowB + T * N;
      const int ng = tile_groups(i);
      for (int gi = 0; gi < ng && ok; ++gi, ++g) {
        const int buf = g & 1;
        if (g >= 2) ok = wait_tm(&tfull[buf], ((g - 2) >> 1) & 1, abort);  // operand buffer free
        if (!ok) break;
        // Items (batch, state group): the group's U x G values of B and of C
        // over the batch, split into three pieces, land in K-rows 3 sg + p of
        // the batch's 16 columns (MN-major: one 16-byte store per 8 columns).
        // Steps past valid_len get zeros (the identity step, [P1] s2.3).
        char* opb = opP + buf * KS * K::OBYTES;
#pragma unroll
        for (int it = 0; it < K::ITEMS / 32; ++it) {
          const int item = it * 32 + lane;
          const int bat = item / NG, sgi = item % NG;  // batch within the group, state group
#pragma unroll
          for (int half = 0; half < 2; ++half) {  // B, then C
            const IO* row = half == 0 ? rowB : rowC;
            float v[8];
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const int s_loc = gi * SPG + bat * U + u;  // step within the tile
              if (s_loc < steps) {
                if constexpr (G == 4) load4<IO>(row + s_loc * N + sgi * G, v + u * G);
                else load8<IO>(row + s_loc * N + sgi * G, v);
              } else {
#pragma unroll
                for (int e = 0; e < G; ++e) v[u * G + e] = 0.f;
              }
            }
            uint4 pcs[3];
            split8(v, pcs);
            const int ngrp = 2 * bat + half;  // 8-column group of the operand
#pragma unroll
            for (int pp = 0; pp < 3; ++pp) {
              const int k = 3 * sgi + pp;  // K-row
              *reinterpret_cast<uint4*>(opb + (k >> 4) * K::OBYTES + ((k >> 3) & 1) * 128 +
                                        ngrp * K::OSBO + (k & 7) * 16) = pcs[pp];
            }
          }
        }
        // K-rows past 3 NG hold zeros: written once per buffer (they never change)
        if (g < 2 && 3 * NG < KS * 16)
          for (int e = lane; e < 32 * (KS * 16 - 3 * NG); e += 32) {
            const int k = 3 * NG + e / 32, ngrp = e % 32;
            *reinterpret_cast<uint4*>(opb + (k >> 4) * K::OBYTES + ((k >> 3) & 1) * 128 +
                                      ngrp * K::OSBO + (k & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (g >= 2) ok = wait_tm(&tempty[buf], ((g - 2) >> 1) & 1, abort);  // TMEM group free
        if (!ok) break;
        if (lane == 0) {
          umma::fence_after_sync();
#pragma unroll
          for (int q = 0; q < KS; ++q) {
            const uint64_t da = umma::smem_desc(umma::smem_u32(opA + q * K::ABYTES), 128, 256);
            const uint64_t dp = umma::smem_desc(umma::smem_u32(opP + (buf * KS + q) * K::OBYTES), 128,
                                                K::OSBO);
            umma::mma_bf16(tbase + buf * 256, da, dp, idesc, q > 0);
          }
          umma::mma_commit(umma::smem_u32(&tfull[buf]));
        }
        __syncwarp();
      }
      if (!ok) break;
      // refill the slot of tile i-1 once every compute warp is done with it
      if (i >= 1 && i - 1 + STAGES < n_tiles) {
        const int ps = (i - 1) % STAGES;
        ok = wait_tm(&empty[ps], ((i - 1) / STAGES) & 1, abort);
        if (ok && lane == 0) issue(i - 1 + STAGES, ps);
        if (ok) ++issued;
      }
    }
    if (!ok) {
      if (lane == 0) atomicOr(la.err, kErrWaitTm);
      // let every copy and product this warp started land before the CTA exits
      for (int i = waited; i < issued; ++i) stream::mbar_wait(&full[i % STAGES], (i / STAGES) & 1);
      if (g >= 1) stream::mbar_wait(&tfull[(g - 1) & 1], ((g - 1) >> 1) & 1);
      if (g >= 2) stream::mbar_wait(&tfull[(g - 2) & 1], ((g - 2) >> 1) & 1);
    }
  } else {
    // ================= compute warps ==============================================
    // Lane (cg, sg): R consecutive channels of channel group cg, the G states
    // of state group sg.  R = 1: f32x2 over pairs of states; R = 2: f32x2 over
    // the pair of channels (the layout of the STREAM tier).
    const int cg = lane / NG, sg = lane % NG;
    const int dw = d0 + warp * CW;        // the warp's first channel
    const int64_t dl = dw + cg * R;       // this lane's first channel
    const bool d_ok = dl < p.dim;         // dim is a multiple of R
    float* pbuf = pbufs + warp * (K::PBYTES / 4);
    const uint32_t tq = tbase + (uint32_t((warp & 3) * 32) << 16);  // this warp's TMEM lanes
    // per-lane constants: log2(e)-scaled A and the initial state, as f32x2
    // pairs (R = 1: states (2q, 2q+1) of the channel; R = 2: state q of the
    // two channels)
    constexpr int NP = R == 1 ? GP : G;
    u64 a2[NP], h2[NP];
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      const int64_t dA = R == 1 ? dl : dl;
      const int64_t dB = R == 1 ? dl : dl + 1;
      const int nA = R == 1 ? sg * G + 2 * q : sg * G + q;
      const int nB = R == 1 ? nA + 1 : nA;
      float lo = 0.f, hi = 0.f, h_lo = 0.f, h_hi = 0.f;
      if (d_ok) {
        lo = __ldg(p.A + dA * N + nA) * kLog2e;
        hi = __ldg(p.A + dB * N + nB) * kLog2e;
        if (p.h0) {  // [P1] s4.1: h_0 = 0 unless given
          h_lo = __ldg(p.h0 + (b * p.dim + dA) * N + nA);
          h_hi = __ldg(p.h0 + (b * p.dim + dB) * N + nB);
        }
      }
      a2[q] = pk2(lo, hi);
      h2[q] = pk2(h_lo, h_hi);
    }
    // the epilogue's view: lane (cp, sl) finishes channels dw + cp R .. + R at
    // steps sl, sl + NG, ... of each block
    constexpr int CG = 32 / NG;
    const int cp = lane % CG, sl = lane / CG;
    const int64_t de = dw + cp * R;
    const bool de_ok = de < p.dim;
    u64 dsk = 0;
    if (de_ok && p.D) dsk = R == 1 ? pk2(__ldg(p.D + de), 0.f) : pk2(__ldg(p.D + de), __ldg(p.D + de + 1));
    IO* __restrict__ yout = static_cast<IO*>(p.y);
    const bool want_states = p.states != nullptr;
    auto chunk_end = [&](int64_t c) { return min((c + 1) * p.chunk_len, L) - 1; };
    int64_t next_c = 0;
    int64_t next_ce = want_states ? chunk_end(0) : INT64_MAX;
    auto put_state = [&](float* dst) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float v[G];
#pragma unroll
        for (int n = 0; n < G; ++n) {
          if constexpr (R == 1) {
            const float2 hv = upk2(h2[n / 2]);
            v[n] = (n & 1) ? hv.y : hv.x;
          } else {
            const float2 hv = upk2(h2[n]);
            v[n] = r ? hv.y : hv.x;
          }
        }
        float* row = dst + (dl + r) * N + sg * G;
#pragma unroll
        for (int k = 0; k < G / 4; ++k)
          *reinterpret_cast<float4*>(row + 4 * k) = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
      }
    };
    auto store_state = [&](int64_t t) {
      if (d_ok) put_state(p.states + (b * p.n_chunks + t / p.chunk_len) * p.dim * N);
    };
    // R values of consecutive channels at element offset e of a slab, as an f32x2 pair
    auto pair_at = [&](const IO* slab, int e) -> u64 {
      if constexpr (R == 1) {
        const float v = widen1<IO>(slab + e);
        return pk2(v, v);
      } else {
        u64 o[1];
        stream::Tile<IO>::template pairs<1>(slab + e, o);
        return o[0];
      }
    };

    bool ok = true;
    int g = 0;  // groups consumed so far
    for (int i = 0; i < n_tiles && ok; ++i) {
      const int slot = i % STAGES;
      char* st = ring + slot * K::STAGE;
      ok = wait_tm(&full[slot], (i / STAGES) & 1, abort);
      if (!ok) break;
      IO* xw = reinterpret_cast<IO*>(st + (0 * W + warp) * K::SLAB);  // the warp's slabs
      IO* dwk = reinterpret_cast<IO*>(st + (1 * W + warp) * K::SLAB);
      const IO* zw = reinterpret_cast<const IO*>(st + (2 * W + warp) * K::SLAB);
      const int64_t t0 = int64_t(i) * T;
      const int steps = tile_steps(i);
      IO* ybase = yout + (b * L + t0) * p.dim + de;
      if (steps < T) {
        // steps past valid_len become the identity (a = 1, b = 0, [P1] s2.3):
        // their delta and x are zeroed (the producer zeroes their B and C)
        for (int e = steps * CW + lane; e < T * CW; e += 32) {
          dwk[e] = IO(0.f);
          xw[e] = IO(0.f);
        }
        __syncwarp();
      }
      const int ng = tile_groups(i);
      for (int gi = 0; gi < ng && ok; ++gi, ++g) {
        const int buf = g & 1;
        ok = wait_tm(&tfull[buf], (g >> 1) & 1, abort);
        if (!ok) break;
        umma::fence_after_sync();
        const int gs0 = gi * SPG;  // first step of the group within the tile
        const uint32_t tcol = tq + buf * 256;
        // One batch of U steps: delta and x of the lane's channels (shared
        // memory, as f32x2 pairs) and the batch's 8 B values (TMEM); its 8 C
        // values are loaded separately, one batch later than B (the recurrence
        // needs C one batch after prepare needs B).
        struct RawB {
          u64 dt[U], x[U];
          TReg<8> b;
        };
        struct RawC {
          TReg<8> c;
        };
        struct Prep {
          u64 ab[U][NP], bi[U][NP];
        };
        constexpr int NBAT = SPG / U;  // batches per group
        // bt: batch within the group; batches past the group re-read its last
        // batch (the values are not used), so no branch splits the loop
        auto clampb = [](int bt) { return bt < NBAT - 1 ? bt : NBAT - 1; };
        auto load_b = [&](RawB& r, int bt) {
          bt = clampb(bt);
          const int s = gs0 + bt * U;
#pragma unroll
          for (int u = 0; u < U; ++u) {
            r.dt[u] = pair_at(dwk, (s + u) * CW + cg * R);
            r.x[u] = pair_at(xw, (s + u) * CW + cg * R);
          }
          tld(tcol + bt * 16, r.b);
        };
        auto load_c = [&](RawC& r, int bt) { tld(tcol + clampb(bt) * 16 + 8, r.c); };
        auto bcval = [](const uint32_t* bc, int i) { return __uint_as_float(bc[i]); };
        auto prepare = [&](Prep& o, const RawB& r) {
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const u64 dd = r.dt[u], uu = mul2(r.dt[u], r.x[u]);  // delta, delta x
            const uint32_t* bv = r.b.r + u * G;
#pragma unroll
            for (int q = 0; q < NP; ++q) {
              const float2 arg = upk2(mul2(dd, a2[q]));
              o.ab[u][q] = pk2(ex2(arg.x), ex2(arg.y));
              const u64 bq = R == 1 ? pk2(bcval(bv, 2 * q), bcval(bv, 2 * q + 1))
                                    : pk2(bcval(bv, q), bcval(bv, q));
              o.bi[u][q] = mul2(uu, bq);
            }
          }
        };
        auto epilogue = [&](int s0) {
          __syncwarp();
#pragma unroll
          for (int e = 0; e < M / NG; ++e) {
            const int j = sl + NG * e;  // step within the block
            const int so = s0 + j;      // step within the tile
            const float* pr = pbuf + j * K::PROW + cp * R;
            float o[R];
            if constexpr (R == 1) {
              float sum = pr[0];
#pragma unroll
              for (int gg = 1; gg < NG; ++gg) sum += pr[gg * K::PS];
              o[0] = fmaf(upk2(dsk).x, widen1<IO>(xw + so * CW + cp), sum);  // + D x
            } else {
              u64 sum = *reinterpret_cast<const u64*>(pr);
#pragma unroll
              for (int gg = 1; gg < NG; ++gg)
                sum = stream::add2(sum, *reinterpret_cast<const u64*>(pr + gg * K::PS));
              u64 xq[1];
              stream::Tile<IO>::template pairs<1>(xw + so * CW + cp * R, xq);
              const float2 yv = upk2(fma2(dsk, xq[0], sum));  // + D x
              o[0] = yv.x;
              o[1] = yv.y;
            }
            if constexpr (K::GATE) {
#pragma unroll
              for (int r = 0; r < R; ++r) o[r] *= silu(widen1<IO>(zw + so * CW + cp * R + r));
            }
            if constexpr (R == 1)
              put1<IO>(ybase + int64_t(so) * p.dim, o[0], de_ok && so < steps);
            else
              stream::Tile<IO>::template put<2>(ybase + int64_t(so) * p.dim, o, de_ok && so < steps);
          }
          __syncwarp();
        };

        RawB rb[2];
        RawC rc[2];
        Prep prep[2];
        load_b(rb[0], 0);
        load_b(rb[1], 1);
        load_c(rc[0], 0);
        tld_wait(rb[0].b, rb[1].b);  // every load complete; the waits tie the registers
        tld_wait(rc[0].c);
        prepare(prep[0], rb[0]);
        const int gend = gs0 + SPG < steps ? gs0 + SPG : steps;  // valid steps of the group end here
        for (int s0 = gs0; s0 < gend; s0 += M) {
          const int64_t b_last = t0 + s0 + M - 1;
          const int bt0 = (s0 - gs0) / U;  // first batch of the block within the group
          auto run_block = [&](auto check) {
            constexpr bool CHECK = decltype(check)::value;
#pragma unroll
            for (int k = 0; k < M / U; ++k) {
              const int s = s0 + k * U;
              // C of batch k+1 and B of batch k+2 are loaded while batch k runs
              // its recurrence and batch k+1 is prepared
              load_c(rc[(k + 1) & 1], bt0 + k + 1);
              load_b(rb[k & 1], bt0 + k + 2);
              const Prep& cur = prep[k & 1];
              const uint32_t* cbat = rc[k & 1].c.r;  // batch k's C values
#pragma unroll
              for (int u = 0; u < U; ++u) {
                const int j = k * U + u;
                constexpr int NA = NP >= 8 ? 4 : (NP >= 4 ? 2 : 1);
                u64 acc[NA];
                const uint32_t* cu = cbat + u * G;
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                  h2[q] = fma2(cur.ab[u][q], h2[q], cur.bi[u][q]);  // h = Abar h + b
                  const u64 cc = R == 1 ? pk2(__uint_as_float(cu[2 * q]), __uint_as_float(cu[2 * q + 1]))
                                        : pk2(__uint_as_float(cu[q]), __uint_as_float(cu[q]));
                  if (q < NA)
                    acc[q] = mul2(cc, h2[q]);
                  else
                    acc[q % NA] = fma2(cc, h2[q], acc[q % NA]);  // C h
                }
#pragma unroll
                for (int a = NA / 2; a >= 1; a /= 2)
#pragma unroll
                  for (int i2 = 0; i2 < a; ++i2) acc[i2] = stream::add2(acc[i2], acc[i2 + a]);
                float* pw = pbuf + j * K::PROW + sg * K::PS + cg * R;
                if constexpr (R == 1) {
                  const float2 a = upk2(acc[0]);
                  *pw = a.x + a.y;
                } else {
                  *reinterpret_cast<u64*>(pw) = acc[0];
                }
                if constexpr (CHECK) {
                  if (t0 + s + u == next_ce) {  // [P1] s3.4 chunk boundary state
                    store_state(next_ce);
                    ++next_c;
                    next_ce = next_c < p.n_chunks ? chunk_end(next_c) : INT64_MAX;
                  }
                }
              }
              prepare(prep[(k + 1) & 1], rb[(k + 1) & 1]);  // batch k+1
              tld_wait(rb[k & 1].b, rc[(k + 1) & 1].c);
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
          epilogue(s0);
        }
        // every TMEM load of the group is complete: hand its columns back
        umma::fence_before_sync();
        __syncwarp();
        if (lane == 0) stream::mbar_arrive(&tempty[buf]);
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) stream::mbar_arrive(&empty[slot]);
    }
    if (!ok) {
      if (lane == 0) atomicOr(la.err, kErrWaitTm);
    } else {
      // steps past valid_len: exact zeros, frozen state for the remaining chunk ends
      if (lv < L) {
        const int64_t total = (L - lv) * CW;
        for (int64_t e = lane; e < total; e += 32) {
          const int64_t t = lv + e / CW;
          const int c = static_cast<int>(e % CW);
          if (dw + c < p.dim) stream::Tile<IO>::put_zero(yout, (b * L + t) * p.dim + dw + c);
        }
      }
      if (want_states)
        for (; next_c < p.n_chunks; ++next_c) store_state(chunk_end(next_c));
      if (p.h_final && d_ok) put_state(p.h_final + b * p.dim * N);
    }
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  if (warp == W) umma::tmem_dealloc(tbase, K::TCOLS);
}

}  // namespace stream_tm
}  // namespace ssm
