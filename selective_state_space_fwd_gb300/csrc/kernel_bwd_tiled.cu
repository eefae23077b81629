// kernel_bwd_tiled.cu -- the backward of the selective scan with TMA-staged
// tiles, for 16, 32 or 64 states and chunks that are a multiple of 16 steps.
//
// The same gradients as the generic backward (kernel_bwd.cu): the adjoint of
// the state runs back over each chunk, replaying the forward from the
// chunk boundary states ([P1] s3.4: the boundary states are kept so that the
// backward recomputes instead of storing every state).  What differs is where
// the data lives:
//
// * Inputs arrive in 16-step tiles by TMA (x, delta, dy, z as [16][channels]
//   of the CTA's channel block; B and C rows as [16][N]), in a ring of stages
//   filled by one thread ahead of the four consuming warps.
// * A first pass over the chunk keeps the state before every 16-step piece in
//   shared memory.  Each piece is then replayed once more with its 16 decays
//   and 17 states held in registers, and the adjoint runs back over it from
//   those registers: the reverse step recomputes no decay (with the gate it
//   still takes the sigmoid of z).
// * dx, d delta and dz of a piece are written to shared-memory tiles and
//   leave by TMA store.
// * dB and dC (sums over channels) are reduced in two levels before any
//   atomic: within the warp, then across the CTA's warps once per piece,
//   ending in one 16-byte vector atomic per four (t, n) per CTA.  The warp
//   sum is a shuffle reduce-scatter over the lane bits that select the
//   channel; with the gate it goes through a transposed shared-memory buffer
//   instead (measured on GB300: the shuffles took fp32 workloads 6-16 % off,
//   but made the bf16 gated ones 2-3 % slower).
//
// Work split: 4 consecutive states per thread (two f32x2 pairs), N / 4
// threads per channel, 128 / N channels per warp, four warps per CTA, all of
// one batch row.
#include <cuda.h>

#include "stream_core.cuh"
#include "tiers.h"

namespace ssm {
namespace bwdt {

using stream::fma2;
using stream::mbar_arrive;
using stream::mbar_expect_tx;
using stream::mbar_init;
using stream::mbar_wait;
using stream::mul2;
using stream::pk2;
using stream::smem_addr;
using stream::tma_load_3d;
using stream::u64;
using stream::upk2;

constexpr int kK = 16;        // steps per tile, per checkpoint and per replayed piece
constexpr int kW = 4;         // warps per CTA
constexpr int kThreads = 32 * kW;
constexpr int kSmemPerSm = 228 * 1024;

// Lane layout with NL lanes per channel: lane l holds state group bwd_sl of
// channel bwd_ch of its warp.  The two lanes of each pair share a state group
// (a warp's 16-byte loads of its B and C slices then cost half the
// shared-memory wavefronts), so a channel's lanes differ in lane bits 1 ..
// log2(NL) and the channels in lane bit 0 and the bits from log2(2 NL) up;
// round r of the warp sum of dB, dC pairs lanes across channel bit
// sum_mask(r).
__host__ __device__ constexpr int bwd_sl(int l, int NL) { return (l >> 1) % NL; }
__host__ __device__ constexpr int bwd_ch(int l, int NL) { return (l / (2 * NL)) * 2 + (l & 1); }
__host__ __device__ constexpr int sum_mask(int r, int NL) { return r == 0 ? 1 : (2 * NL) << (r - 1); }
// The layout gives each (channel, state group) to one lane, and the LCW
// rounds pair lanes of one state group and different channels, reaching every
// channel of the warp.
constexpr bool sum_masks_ok(int NL, int LCW) {
  const int CW = 32 / NL;
  bool seen[32] = {};
  for (int l = 0; l < 32; ++l) {
    const int sl = bwd_sl(l, NL), ch = bwd_ch(l, NL);
    if (sl >= NL || ch >= CW || seen[ch * NL + sl]) return false;
    seen[ch * NL + sl] = true;
    bool reach[32] = {};
    for (int sub = 0; sub < (1 << LCW); ++sub) {
      int p = l;
      for (int r = 0; r < LCW; ++r)
        if (sub >> r & 1) p ^= sum_mask(r, NL);
      if (p < 0 || p >= 32 || bwd_sl(p, NL) != sl) return false;
      reach[bwd_ch(p, NL)] = true;
    }
    for (int c = 0; c < CW; ++c)
      if (!reach[c]) return false;
  }
  return true;
}

template <int N_, typename T_, bool GATE_, bool RANK_ = false>
struct Cfg {
  static constexpr int N = N_;
  using T = T_;
  static constexpr bool GATE = GATE_;
  // RANK: rows with valid lengths taken longest first (rows_ranked, row_of_rank)
  static constexpr bool RANK = RANK_;
  static constexpr int G = 4;              // states per thread
  static constexpr int NL = N / G;         // threads per channel
  static constexpr int CWB = 32 / NL;      // channels per warp
  static constexpr int CPB = CWB * kW;     // channels per CTA
  static constexpr int ES = sizeof(T);
  static constexpr int ACT = kK * CPB * ES;  // one activation tile
  static constexpr int ROW = kK * N * ES;    // one tile of B or C rows
  static constexpr int NACT = GATE ? 4 : 3;  // x, delta, dy (, z)
  static constexpr int STAGE = NACT * ACT + 2 * ROW;
  static constexpr int TX1 = 2 * ACT + ROW;  // checkpoint pass: x, delta, B
  static constexpr int TX2 = STAGE;          // pieces: everything
  static constexpr int NOUT = GATE ? 3 : 2;  // dx, d delta (, dz)
  static constexpr int OUTB = kK * CPB * ES;
  static constexpr int OPL = 2 * N / 32;     // dB/dC outputs per lane in the warp sum
  static constexpr int LCW = CWB == 8 ? 3 : (CWB == 4 ? 2 : 1);  // log2 of the channels per warp
  static constexpr bool XPOSE = GATE;        // warp sum through the transpose buffer
  static constexpr int XS = 2 * N + 16;      // row stride (floats) of the transpose buffer
  static constexpr int XBUF = XPOSE ? CWB * XS * 4 : 0;  // bytes per warp
  static constexpr int REDB = kK * kW * 2 * N * 4;
  static_assert(N % 16 == 0 && N <= 64, "16, 32 or 64 states");
  static_assert(ACT % 128 == 0 && ROW % 128 == 0 && XBUF % 128 == 0, "tile alignment");
  static_assert((1 << LCW) == CWB && 8 >> LCW == OPL, "warp sum of dB, dC");
  static_assert(sum_masks_ok(NL, LCW), "lane layout and the masks of the warp sum");
};

// Shared memory of a CTA: the ring, the checkpoints (one 16-byte slot per
// thread and piece), the output tiles, the warps' transpose buffers (gate
// instances), the CTA's dB/dC partial sums, the mbarriers.
template <class K>
size_t smem_bytes(int stages, int nck) {
  return size_t(stages) * K::STAGE + size_t(nck) * kThreads * 16 + K::NOUT * K::OUTB +
         kW * K::XBUF + K::REDB + 2 * stages * sizeof(uint64_t);
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, int c0, int c1, int c2,
                                             const void* src) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(src))
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Element access of the staged tiles.
__device__ __forceinline__ float f32_of(float v) { return v; }
__device__ __forceinline__ float f32_of(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ void put(float* p, float v) { *p = v; }
__device__ __forceinline__ void put(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
// Four consecutive values of a B or C row as two fp32 pairs.
__device__ __forceinline__ void row4(const float* p, u64& lo, u64& hi) {
  const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(p);
  lo = v.x;
  hi = v.y;
}
__device__ __forceinline__ void row4(const __nv_bfloat16* p, u64& lo, u64& hi) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
  lo = pk2(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u));
  hi = pk2(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
}
__device__ __forceinline__ float hsum(u64 v) {
  const float2 f = upk2(v);
  return f.x + f.y;
}

// The order in which a CTA consumes tiles: chunks newest first; in each chunk
// the checkpoint pass over pieces 0 .. nt-2, then the pieces nt-1 .. 0.  The
// filling thread walks the same order ahead of the consumers.
struct TileSeq {
  int64_t c, j, nt, CL, L, lv;
  int phase;  // 0: checkpoint pass, 1: pieces
  __device__ void start_chunk() {
    for (; c >= 0; --c) {
      const int64_t t0 = c * CL, t1 = min(t0 + CL, L), tv = min(t1, lv);
      if (tv > t0) {
        nt = (tv - t0 + kK - 1) / kK;
        phase = nt > 1 ? 0 : 1;
        j = phase == 0 ? 0 : nt - 1;
        return;
      }
    }
  }
  __device__ bool next(int64_t& s0, int& kind) {
    if (c < 0) return false;
    s0 = c * CL + j * kK;
    kind = phase;
    if (phase == 0) {
      if (++j >= nt - 1) {
        phase = 1;
        j = nt - 1;
      }
    } else if (--j < 0) {
      --c;
      start_chunk();
    }
    return true;
  }
};

struct Maps {
  CUtensorMap x, dt, dy, z, b, c, dx, ddt, dz;
};

template <class K>
__global__ void __launch_bounds__(kThreads, 2)
    bwd_tiled_kernel(const __grid_constant__ Maps m, const BwdParams p, const int stages,
                     unsigned int* err) {
  constexpr int N = K::N, NL = K::NL, CWB = K::CWB, CPB = K::CPB;
  using T = typename K::T;
  extern __shared__ __align__(128) char smem[];
  const int S = stages;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t L = p.fwd.seqlen, D_ = p.fwd.dim, CL = p.fwd.chunk_len;
  const int nck = static_cast<int>(CL / kK);
  char* ring = smem;
  float4* ck = reinterpret_cast<float4*>(smem + S * K::STAGE);
  char* outs = smem + S * K::STAGE + size_t(nck) * kThreads * 16;
  T* o_dx = reinterpret_cast<T*>(outs);
  T* o_ddt = reinterpret_cast<T*>(outs + K::OUTB);
  T* o_dz = reinterpret_cast<T*>(outs + 2 * K::OUTB);
  float* xbuf = reinterpret_cast<float*>(outs + K::NOUT * K::OUTB + warp * K::XBUF);
  float* red = reinterpret_cast<float*>(outs + K::NOUT * K::OUTB + kW * K::XBUF);
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<char*>(red) + K::REDB);
  uint64_t* empty = full + S;

  const int64_t nblk = (D_ + CPB - 1) / CPB;
  const int b = static_cast<int>(K::RANK && rows_ranked(p.fwd) ? row_of_rank(p.fwd, blockIdx.x / nblk)
                                                                : blockIdx.x / nblk);
  const int d0 = static_cast<int>((blockIdx.x % nblk) * CPB);
  const int sl = bwd_sl(lane, NL), ch = bwd_ch(lane, NL), n0 = sl * 4;  // lane layout above
  const int cc = warp * CWB + ch;  // the thread's channel within the CTA's block
  const bool ok = d0 + cc < D_;
  const int64_t dd = ok ? d0 + cc : 0;
  const int64_t lv = valid_steps(p.fwd, b);
  const int64_t nch = (L + CL - 1) / CL;

  // Steps past the valid length beyond the last partly valid piece: zero
  // gradients (the partly valid piece writes its own zeros).
  {
    const int64_t z0 = min((lv + kK - 1) / kK * kK, L);
    const int64_t total = (L - z0) * CPB;
    for (int64_t e = tid; e < total; e += kThreads) {
      const int64_t t = z0 + e / CPB;
      const int c = static_cast<int>(e % CPB);
      if (d0 + c < D_) {
        const int64_t i = (b * L + t) * D_ + d0 + c;
        put(static_cast<T*>(p.dx) + i, 0.f);
        put(static_cast<T*>(p.ddelta) + i, 0.f);
        if (K::GATE) put(static_cast<T*>(p.dz) + i, 0.f);
      }
    }
  }

  TileSeq seq;
  int64_t issued = 0;
  auto issue = [&](int slot, int64_t s0, int kind) {
    char* st = ring + slot * K::STAGE;
    const int t = static_cast<int>(s0);
    mbar_expect_tx(&full[slot], kind == 0 ? K::TX1 : K::TX2);
    tma_load_3d(st, &m.x, d0, t, b, &full[slot]);
    tma_load_3d(st + K::ACT, &m.dt, d0, t, b, &full[slot]);
    tma_load_3d(st + K::NACT * K::ACT, &m.b, 0, t, b, &full[slot]);
    if (kind == 1) {
      tma_load_3d(st + 2 * K::ACT, &m.dy, d0, t, b, &full[slot]);
      if constexpr (K::GATE) tma_load_3d(st + 3 * K::ACT, &m.z, d0, t, b, &full[slot]);
      tma_load_3d(st + K::NACT * K::ACT + K::ROW, &m.c, 0, t, b, &full[slot]);
    }
    ++issued;
  };
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kW);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    seq.c = nch - 1;
    seq.CL = CL;
    seq.L = L;
    seq.lv = lv;
    seq.start_chunk();
    int64_t s0;
    int kind;
    for (int s = 0; s < S && seq.next(s0, kind); ++s) issue(s, s0, kind);
  }
  __syncthreads();

  // A of the thread's states (pairs), and scaled by log2(e) for ex2.
  u64 A2[2], AL2[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const float a0 = ok ? __ldg(p.fwd.A + dd * N + n0 + 2 * q) : 0.f;
    const float a1 = ok ? __ldg(p.fwd.A + dd * N + n0 + 2 * q + 1) : 0.f;
    A2[q] = pk2(a0, a1);
    AL2[q] = pk2(a0 * kLog2e, a1 * kLog2e);
  }
  const float dsk = (ok && p.fwd.D) ? __ldg(p.fwd.D + dd) : 0.f;
  u64 lam2[2], dacc2[2];
  lam2[0] = lam2[1] = dacc2[0] = dacc2[1] = pk2(0.f, 0.f);
  float dDacc = 0.f;

  uint32_t it = 0;  // tiles consumed
  bool good = true;
  auto acquire = [&]() -> const char* {
    const int s = static_cast<int>(it % S);
    if (good && !mbar_wait(&full[s], (it / S) & 1)) good = false;
    if (tid == 0 && it >= 1 && good) {  // refill the stage the previous tile used
      const int ps = static_cast<int>((it - 1) % S);
      if (!mbar_wait(&empty[ps], ((it - 1) / S) & 1)) {
        good = false;
      } else {
        int64_t s0;
        int kind;
        if (seq.next(s0, kind)) issue(ps, s0, kind);
      }
    }
    return ring + s * K::STAGE;
  };
  auto release = [&]() {
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[it % S]);
    ++it;
  };

  for (int64_t c = nch - 1; c >= 0 && good; --c) {
    const int64_t t0 = c * CL, t1 = min(t0 + CL, L), tv = min(t1, lv);
    if (tv <= t0) continue;
    const int nt = static_cast<int>((tv - t0 + kK - 1) / kK);
    u64 h2[2];
    {
      float4 h = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ok) {
        if (c > 0)
          h = *reinterpret_cast<const float4*>(
              p.fwd.states + ((b * p.fwd.n_chunks + c - 1) * D_ + dd) * N + n0);
        else if (p.fwd.h0)
          h = *reinterpret_cast<const float4*>(p.fwd.h0 + (b * D_ + dd) * N + n0);
      }
      h2[0] = pk2(h.x, h.y);
      h2[1] = pk2(h.z, h.w);
    }
    // checkpoint pass: the forward over pieces 0 .. nt-2, the state before
    // each piece kept in this thread's slot
    for (int j = 0; j < nt - 1; ++j) {
      const char* st = acquire();
      {
        const float2 lo = upk2(h2[0]), hi = upk2(h2[1]);
        ck[j * kThreads + tid] = make_float4(lo.x, lo.y, hi.x, hi.y);
      }
      const T* xs = reinterpret_cast<const T*>(st) + cc;
      const T* ds = reinterpret_cast<const T*>(st + K::ACT) + cc;
      const T* bs = reinterpret_cast<const T*>(st + K::NACT * K::ACT) + n0;
#pragma unroll
      for (int k = 0; k < kK; ++k) {
        const float dt = f32_of(ds[k * CPB]), ux = dt * f32_of(xs[k * CPB]);
        u64 B2[2];
        row4(bs + k * N, B2[0], B2[1]);
        const u64 dt2 = pk2(dt, dt), ux2 = pk2(ux, ux);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float2 arg = upk2(mul2(dt2, AL2[q]));
          h2[q] = fma2(pk2(ex2(arg.x), ex2(arg.y)), h2[q], mul2(ux2, B2[q]));
        }
      }
      release();
    }
    {
      const float2 lo = upk2(h2[0]), hi = upk2(h2[1]);
      ck[(nt - 1) * kThreads + tid] = make_float4(lo.x, lo.y, hi.x, hi.y);
    }
    // the pieces, newest first
    for (int j = nt - 1; j >= 0; --j) {
      const char* st = acquire();
      const int64_t s0 = t0 + int64_t(j) * kK;
      const int len = static_cast<int>(min(int64_t(kK), tv - s0));
      if (len < kK) {
        // steps of the piece past the valid length read as zeros (identity
        // steps with no output); the stage is refilled by TMA afterwards
        char* w = const_cast<char*>(st);
        auto zero_rows = [&](int off, int inner) {
          const int lo = (len * inner * K::ES) / 4, hi = (kK * inner * K::ES) / 4;
          uint32_t* u = reinterpret_cast<uint32_t*>(w + off);
          for (int i = lo + tid; i < hi; i += kThreads) u[i] = 0u;
        };
        for (int a = 0; a < K::NACT; ++a) zero_rows(a * K::ACT, CPB);
        zero_rows(K::NACT * K::ACT, N);
        zero_rows(K::NACT * K::ACT + K::ROW, N);
        fence_async_smem();
        __syncthreads();
      }
      const T* xs = reinterpret_cast<const T*>(st) + cc;
      const T* ds = reinterpret_cast<const T*>(st + K::ACT) + cc;
      const T* ys = reinterpret_cast<const T*>(st + 2 * K::ACT) + cc;
      const T* zs = reinterpret_cast<const T*>(st + 3 * K::ACT) + cc;
      const T* bs = reinterpret_cast<const T*>(st + K::NACT * K::ACT) + n0;
      const T* cs = bs + kK * N;
      // replay: the piece's decays and states, in registers
      u64 a2[kK][2], hs[kK + 1][2];
      {
        const float4 h = ck[j * kThreads + tid];
        hs[0][0] = pk2(h.x, h.y);
        hs[0][1] = pk2(h.z, h.w);
      }
#pragma unroll
      for (int k = 0; k < kK; ++k) {
        const float dt = f32_of(ds[k * CPB]), ux = dt * f32_of(xs[k * CPB]);
        u64 B2[2];
        row4(bs + k * N, B2[0], B2[1]);
        const u64 dt2 = pk2(dt, dt), ux2 = pk2(ux, ux);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float2 arg = upk2(mul2(dt2, AL2[q]));
          a2[k][q] = pk2(ex2(arg.x), ex2(arg.y));
          hs[k + 1][q] = fma2(a2[k][q], hs[k][q], mul2(ux2, B2[q]));
        }
      }
      // the adjoint back over the piece.  A step's inputs are loaded one step
      // ahead (before the previous step's warp barrier, which the compiler
      // does not move loads across), so their shared-memory latency overlaps
      // that step's arithmetic.
      struct In {
        float dt, x, dy, z;
        u64 B2[2], C2[2];
      };
      auto load_in = [&](int k) {
        In v;
        v.dt = f32_of(ds[k * CPB]);
        v.x = f32_of(xs[k * CPB]);
        v.dy = f32_of(ys[k * CPB]);
        v.z = K::GATE ? f32_of(zs[k * CPB]) : 0.f;
        row4(bs + k * N, v.B2[0], v.B2[1]);
        row4(cs + k * N, v.C2[0], v.C2[1]);
        return v;
      };
      In nxt = load_in(kK - 1);
#pragma unroll
      for (int k = kK - 1; k >= 0; --k) {
        const In cur = nxt;
        if (k > 0) nxt = load_in(k - 1);
        const float dt = cur.dt, x = cur.x, dy = cur.dy;
        const u64(&B2)[2] = cur.B2;
        const u64(&C2)[2] = cur.C2;
        float dyp = dy, z = 0.f, sg = 0.f;
        if constexpr (K::GATE) {
          z = cur.z;
          sg = __fdividef(1.f, 1.f + ex2(-z * kLog2e));
          dyp = dy * z * sg;  // dy silu(z)
        }
        const float ux = dt * x;
        const u64 dyp2 = pk2(dyp, dyp), dt2 = pk2(dt, dt), ux2 = pk2(ux, ux);
        const u64 zero2 = pk2(0.f, 0.f);
        u64 pA2 = zero2, S12 = zero2, yp2 = zero2, db2[2], dc2[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          lam2[q] = fma2(C2[q], dyp2, lam2[q]);      // + C_t dyp_t
          const u64 r2 = mul2(lam2[q], mul2(a2[k][q], hs[k][q]));  // lambda a_t h_{t-1}
          pA2 = fma2(A2[q], r2, pA2);
          dacc2[q] = fma2(dt2, r2, dacc2[q]);
          S12 = fma2(lam2[q], B2[q], S12);
          db2[q] = mul2(lam2[q], ux2);
          dc2[q] = mul2(dyp2, hs[k + 1][q]);
          if constexpr (K::GATE) yp2 = fma2(C2[q], hs[k + 1][q], yp2);
          lam2[q] = mul2(lam2[q], a2[k][q]);         // carried to step t - 1
        }
        float pA = hsum(pA2), S1 = hsum(S12), yp = hsum(yp2);
#pragma unroll
        for (int msk = 2; msk < 2 * NL; msk *= 2) {  // over the channel's lanes
          pA += __shfl_xor_sync(0xffffffffu, pA, msk);
          S1 += __shfl_xor_sync(0xffffffffu, S1, msk);
          if constexpr (K::GATE) yp += __shfl_xor_sync(0xffffffffu, yp, msk);
        }
        float g_dt = fmaf(x, S1, pA), g_dx = fmaf(dt, S1, dsk * dyp), g_dz = 0.f;
        if constexpr (K::GATE) {
          yp = fmaf(dsk, x, yp);  // C h + D x, before the gate
          g_dz = dy * yp * sg * (1.f + z * (1.f - sg));
        }
        dDacc = fmaf(dyp, x, dDacc);
        if (k >= len) g_dt = g_dx = g_dz = 0.f;
        if (sl == 0) {
          put(o_dx + k * CPB + cc, g_dx);
          put(o_ddt + k * CPB + cc, g_dt);
          if constexpr (K::GATE) put(o_dz + k * CPB + cc, g_dz);
        }
        // dB, dC summed over the warp's channels by a reduce-scatter: in each
        // round over one channel bit of the lane (lane bit 0, then the bits
        // from log2(2 NL) up) a lane keeps one half of its values, adds the
        // partner's copy of that half and hands over the other half.  The
        // lane ends with OPL outputs of its state group, from position o of
        // (dB n0 .. n0+3, dC n0 .. n0+3).
        if constexpr (K::XPOSE) {
          // through the transpose buffer: each lane stores its four of each,
          // then lane o sums output o (and o + 32, ...) over the channels
          const float2 b0 = upk2(db2[0]), b1 = upk2(db2[1]);
          const float2 c0 = upk2(dc2[0]), c1 = upk2(dc2[1]);
          *reinterpret_cast<float4*>(xbuf + ch * K::XS + n0) = make_float4(b0.x, b0.y, b1.x, b1.y);
          *reinterpret_cast<float4*>(xbuf + ch * K::XS + N + n0) =
              make_float4(c0.x, c0.y, c1.x, c1.y);
          __syncwarp();
#pragma unroll
          for (int o = 0; o < K::OPL; ++o) {
            float v[CWB];  // summed as a tree: short dependency chains
#pragma unroll
            for (int c2 = 0; c2 < CWB; ++c2) v[c2] = xbuf[c2 * K::XS + lane + 32 * o];
#pragma unroll
            for (int w = CWB / 2; w >= 1; w /= 2)
#pragma unroll
              for (int i = 0; i < w; ++i) v[i] += v[i + w];
            red[(k * kW + warp) * 2 * N + lane + 32 * o] = v[0];
          }
          __syncwarp();
        } else {
          const float2 b0 = upk2(db2[0]), b1 = upk2(db2[1]);
          const float2 c0 = upk2(dc2[0]), c1 = upk2(dc2[1]);
          float v[8] = {b0.x, b0.y, b1.x, b1.y, c0.x, c0.y, c1.x, c1.y};
          int o = 0;
#pragma unroll
          for (int r = 0; r < K::LCW; ++r) {
            const int w = 8 >> r, m = sum_mask(r, NL);
            const bool hi = (lane & m) != 0;
#pragma unroll
            for (int i = 0; i < w / 2; ++i) {
              const float give = hi ? v[i] : v[i + w / 2];
              const float keep = hi ? v[i + w / 2] : v[i];
              v[i] = keep + __shfl_xor_sync(0xffffffffu, give, m);
            }
            o += hi ? w / 2 : 0;
          }
#pragma unroll
          for (int j = 0; j < K::OPL; ++j) {
            const int q = o + j;  // 0..3: dB of state n0 + q; 4..7: dC of state n0 + q - 4
            red[(k * kW + warp) * 2 * N + (q < 4 ? n0 + q : N + n0 + q - 4)] = v[j];
          }
        }
      }
      fence_async_smem();  // the output tiles go out by TMA
      release();
      if (__syncthreads_or(!good)) {
        good = false;
        break;
      }
      if (tid == 0) {
        tma_store_3d(&m.dx, d0, static_cast<int>(s0), b, o_dx);
        tma_store_3d(&m.ddt, d0, static_cast<int>(s0), b, o_ddt);
        if constexpr (K::GATE) tma_store_3d(&m.dz, d0, static_cast<int>(s0), b, o_dz);
        bulk_commit();
      }
      // the CTA's dB, dC: the warps' sums added, one vector atomic per four
      constexpr int Q = 2 * N / 4;  // float4 groups per step
      for (int g = tid; g < kK * Q; g += kThreads) {
        const int k = g / Q, o = (g % Q) * 4;
        const int64_t t = s0 + k;
        if (t >= tv) continue;
        float4 v = *reinterpret_cast<const float4*>(red + (k * kW) * 2 * N + o);
#pragma unroll
        for (int w = 1; w < kW; ++w) {
          const float4 u = *reinterpret_cast<const float4*>(red + (k * kW + w) * 2 * N + o);
          v.x += u.x;
          v.y += u.y;
          v.z += u.z;
          v.w += u.w;
        }
        float* dst = o < N ? p.dB + (b * L + t) * N + o : p.dC + (b * L + t) * N + (o - N);
        atomicAdd(reinterpret_cast<float4*>(dst), v);
      }
      if (tid == 0) bulk_wait_read();  // the output tiles are free again
      __syncthreads();
    }
  }
  if (!good) {
    if (lane == 0) atomicOr(err, stream::kErrWait);
    if (tid == 0) {
      // let the copies already issued land before the CTA's memory is released
      for (int64_t i = it; i < issued; ++i)
        mbar_wait(&full[i % S], static_cast<uint32_t>((i / S) & 1));
      bulk_wait_all();
    }
    return;
  }
  if (tid == 0) bulk_wait_all();
  if (ok) {
    const float2 a0 = upk2(dacc2[0]), a1 = upk2(dacc2[1]);
    atomicAdd(reinterpret_cast<float4*>(p.dA + dd * N + n0), make_float4(a0.x, a0.y, a1.x, a1.y));
    if (p.dh0) {
      const float2 l0 = upk2(lam2[0]), l1 = upk2(lam2[1]);
      *reinterpret_cast<float4*>(p.dh0 + (b * D_ + dd) * N + n0) =
          make_float4(l0.x, l0.y, l1.x, l1.y);
    }
    if (sl == 0 && p.dD) atomicAdd(p.dD + dd, dDacc);
  }
}

int smem_limit_per_cta() { return 227 * 1024; }

// Ring depth: the deepest of 4, 3, 2 that keeps two CTAs per SM, else the
// deepest that fits one.
template <class K>
int pick_stages(int nck) {
  for (int s = 4; s >= 2; --s)
    if (2 * (smem_bytes<K>(s, nck) + 1024) <= size_t(kSmemPerSm)) return s;
  for (int s = 4; s >= 2; --s)
    if (smem_bytes<K>(s, nck) <= size_t(smem_limit_per_cta())) return s;
  return 0;
}

template <class K>
cudaError_t launch_k(const BwdParams& p, cudaStream_t s) {
  const bool bf16 = K::ES == 2;
  const ScanParams& f = p.fwd;
  Maps m;
  if (!stream::make_map(&m.x, f.x, bf16, f.dim, f.seqlen, f.batch, K::CPB, kK) ||
      !stream::make_map(&m.dt, f.delta, bf16, f.dim, f.seqlen, f.batch, K::CPB, kK) ||
      !stream::make_map(&m.dy, p.dy, bf16, f.dim, f.seqlen, f.batch, K::CPB, kK) ||
      !stream::make_map(&m.b, f.B, bf16, K::N, f.seqlen, f.batch, K::N, kK) ||
      !stream::make_map(&m.c, f.C, bf16, K::N, f.seqlen, f.batch, K::N, kK) ||
      !stream::make_map(&m.dx, p.dx, bf16, f.dim, f.seqlen, f.batch, K::CPB, kK) ||
      !stream::make_map(&m.ddt, p.ddelta, bf16, f.dim, f.seqlen, f.batch, K::CPB, kK))
    return cudaErrorInvalidValue;
  if constexpr (K::GATE) {
    if (!stream::make_map(&m.z, f.z, bf16, f.dim, f.seqlen, f.batch, K::CPB, kK) ||
        !stream::make_map(&m.dz, p.dz, bf16, f.dim, f.seqlen, f.batch, K::CPB, kK))
      return cudaErrorInvalidValue;
  } else {
    m.z = m.x;  // unused
    m.dz = m.dx;
  }
  const int nck = static_cast<int>(f.chunk_len / kK);
  const int stages = pick_stages<K>(nck);
  if (stages == 0) return cudaErrorInvalidValue;
  const size_t smem = smem_bytes<K>(stages, nck);
  unsigned int* err = stream::error_word();
  if (err == nullptr) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(bwd_tiled_kernel<K>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem_limit_per_cta());
  if (e != cudaSuccess) return e;
  const int64_t blocks = (f.dim + K::CPB - 1) / K::CPB * f.batch;
  bwd_tiled_kernel<K><<<static_cast<unsigned>(blocks), kThreads, smem, s>>>(m, p, stages, err);
  return cudaGetLastError();
}

template <typename T, bool GATE>
cudaError_t launch_tg(const BwdParams& p, cudaStream_t s) {
  // rows with valid lengths run longest first (the host side of rows_ranked)
  const bool rank = p.fwd.valid_len != nullptr && p.fwd.batch <= 32;
  switch (p.fwd.dstate) {
    case 16: return rank ? launch_k<Cfg<16, T, GATE, true>>(p, s) : launch_k<Cfg<16, T, GATE>>(p, s);
    case 32: return rank ? launch_k<Cfg<32, T, GATE, true>>(p, s) : launch_k<Cfg<32, T, GATE>>(p, s);
    case 64: return rank ? launch_k<Cfg<64, T, GATE, true>>(p, s) : launch_k<Cfg<64, T, GATE>>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

template <class K>
size_t smem_for(int nck) {
  const int st = pick_stages<K>(nck);
  return st == 0 ? SIZE_MAX : smem_bytes<K>(st, nck);
}

template <typename T, bool GATE>
size_t smem_tg(int n, int nck) {
  switch (n) {
    case 16: return smem_for<Cfg<16, T, GATE>>(nck);
    case 32: return smem_for<Cfg<32, T, GATE>>(nck);
    case 64: return smem_for<Cfg<64, T, GATE>>(nck);
    default: return SIZE_MAX;
  }
}

size_t smem_of(int n, bool bf16, bool gate, int nck) {
  if (bf16) return gate ? smem_tg<__nv_bfloat16, true>(n, nck) : smem_tg<__nv_bfloat16, false>(n, nck);
  return gate ? smem_tg<float, true>(n, nck) : smem_tg<float, false>(n, nck);
}

}  // namespace bwdt

bool bwd_tiled_eligible(const BwdParams& p, bool bf16) {
  const ScanParams& f = p.fwd;
  const int N = f.dstate;
  if (N != 16 && N != 32 && N != 64) return false;
  if (f.chunk_len <= 0 || f.chunk_len % bwdt::kK != 0) return false;
  const int es = bf16 ? 2 : 4;
  if ((f.dim * es) % 16 != 0) return false;
  if (f.seqlen > INT32_MAX || f.batch > INT32_MAX || f.dim > INT32_MAX / 2) return false;
  const uintptr_t mis =
      reinterpret_cast<uintptr_t>(f.x) | reinterpret_cast<uintptr_t>(f.delta) |
      reinterpret_cast<uintptr_t>(f.B) | reinterpret_cast<uintptr_t>(f.C) |
      reinterpret_cast<uintptr_t>(f.z) | reinterpret_cast<uintptr_t>(f.states) |
      reinterpret_cast<uintptr_t>(f.h0) | reinterpret_cast<uintptr_t>(p.dy) |
      reinterpret_cast<uintptr_t>(p.dx) | reinterpret_cast<uintptr_t>(p.ddelta) |
      reinterpret_cast<uintptr_t>(p.dz) | reinterpret_cast<uintptr_t>(p.dA) |
      reinterpret_cast<uintptr_t>(p.dB) | reinterpret_cast<uintptr_t>(p.dC) |
      reinterpret_cast<uintptr_t>(p.dh0);
  if (mis % 16 != 0) return false;
  if (!stream::tma_encode_available()) return false;
  const int nck = static_cast<int>(f.chunk_len / bwdt::kK);
  return bwdt::smem_of(N, bf16, f.z != nullptr, nck) <= size_t(bwdt::smem_limit_per_cta());
}

cudaError_t launch_bwd_tiled(const BwdParams& p, bool bf16, cudaStream_t s) {
  if (bf16)
    return p.fwd.z ? bwdt::launch_tg<__nv_bfloat16, true>(p, s)
                   : bwdt::launch_tg<__nv_bfloat16, false>(p, s);
  return p.fwd.z ? bwdt::launch_tg<float, true>(p, s) : bwdt::launch_tg<float, false>(p, s);
}

}  // namespace ssm
