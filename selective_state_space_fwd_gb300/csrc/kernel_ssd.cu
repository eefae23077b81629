// kernel_ssd.cu -- the SSD form of the scan (one decay per head) on the
// tensor cores ([P2] s5.1-s5.2: the recurrence expanded into a semiseparable
// matrix product; blocks of steps done as matrix products, the state carried
// from block to block by the recurrence itself).
//
// Per head h with decay a_t = exp(delta_t A_h) and a block of Q = 128 steps,
// write cs_t = sum_{r<=t} delta_r A_h (in log2 units) inside the block,
// e_s = cs_s - log2(delta_s) and S for the state entering the block ([N x P]:
// state n, channel p of the head):
//   G[t,s]  = C_t . B_s                                     (tensor cores, K = N)
//   Ym[t,s] = G[t,s] 2^(cs_t - e_s) for s <= t, else 0      (registers)
//   Yd      = Ym x                                          (tensor cores, K = Q)
//   Yo      = C S                                           (tensor cores, K = N)
//   y_t     = (Yd_t + 2^cs_t Yo_t + D x_t) silu(z_t)
//   S      <- 2^cs_end S + B^T (delta_s 2^(cs_end - cs_s) x_s)   (tensor cores, K = Q)
// which is the recurrence regrouped: the output of step t is the inputs of
// the block weighted by the decay between their step and t, plus the state
// entering the block decayed to t.  Operands are bf16 in shared memory,
// products accumulate in fp32 in tensor memory.  The state stays fp32 in
// tensor memory between blocks: before the products of a block each thread
// reads its state row (rounded to bf16 as the operand of Yo) and writes it
// back scaled by 2^cs_end, and the state-update product accumulates onto it.
//
// One CTA of 256 threads per (batch row, head), blocks in order.  The C, B
// and x tiles of a block arrive by TMA as 128-byte swizzled boxes; the C copy
// of the next block starts once the first products are done with C, the B
// and x copies once the second is.  Threads i and i + 128 share row i: step
// i of the block for the masked block matrix and the epilogue (TMEM lane i
// holds row i of G, Yd and Yo) and state row i (and i + 128 with 256 states;
// lane i of S), each taking half of the columns (warps w and w + 4 read the
// same TMEM lanes).  With 128 states shared memory is about 115 KB, so two
// CTAs share an SM and one CTA's staging and epilogue overlap the other's
// matrix products; with 256 states (C and B tiles of 64 KB) one CTA fits.
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "ssd.h"
#include "umma.cuh"

namespace ssm {
namespace {

constexpr int Q = kSsdChunk, P = kSsdHeadDim;
constexpr int kThreads = 128;  // rows of a block; the CTA has two threads per row
constexpr unsigned kSsdWaitLimit = 1u << 24;  // try_wait polls before a wait gives up
constexpr unsigned kErrSsdWait = 2u;
constexpr unsigned kErrSsdAlign = 4u;  // shared memory not 1024-byte aligned: nothing computed

// Two tile layouts.  The tiles that arrive by TMA (C, B, x) are 128-byte
// swizzled: 64 bf16 of each of the 128 rows per 16 KB part, row r at r * 128,
// its 16-byte chunk c stored at chunk c ^ (r mod 8), in 1024-byte atoms of 8
// rows (the pattern the TMA writes and the tensor core reads).  The tiles that
// threads write (Xw, S, Ym) are column strips: strip c holds 16 bytes (8 bf16)
// of each row, row r at c * (strip size) + r * 16; core matrix (r8, c) then
// sits at c * (strip size) + r8 * 128, a K-major operand when the strips run
// along K and an MN-major one when they run along M/N.
constexpr uint32_t kStrip = Q * 16;   // a strip of 128 rows
constexpr uint32_t kHalf = Q * 128;   // one 64-column part of a swizzled tile

// Layout for NS states: C and B tiles of NS / 64 swizzled parts, the state
// tile [p x n] in strips of NS rows; TMEM holds NS / 128 state rows per lane.
template <int NS>
struct SsdCfg {
  static_assert(NS == 128 || NS == 256, "128 or 256 states");
  static constexpr int N = NS;
  static constexpr int NQ = N / 64;   // 64-column parts of the C and B tiles
  static constexpr int NH = N / 128;  // state rows per TMEM lane (row n, n + 128)
  static constexpr uint32_t kStripS = N * 16;
  static constexpr uint32_t kTileC = 0;                    // C rows [t x n], swizzled parts
  static constexpr uint32_t kTileB = kTileC + N * Q * 2;   // B rows [s x n], as C; then Ym [t x s]
  static constexpr uint32_t kTileX = kTileB + N * Q * 2;   // x rows [s x p], swizzled
  static constexpr uint32_t kTileXw = kTileX + P * Q * 2;  // delta_s 2^(cs_end - cs_s) x_s, strips
  static constexpr uint32_t kTileS = kTileXw + P * Q * 2;  // state rows [n x p], strips of N rows
  static constexpr uint32_t kDs = kTileS + P * N * 2;      // D of the head's channels, fp32 [P]
  static constexpr uint32_t kWarpTot = kDs + P * 4;        // per-warp totals of the scan of cs
  static constexpr uint32_t kBar = kWarpTot + 16;          // mbarrier of the matrix products
  static constexpr uint32_t kTBar = kBar + 8;              // mbarrier of the TMA copies
  static constexpr uint32_t kSlot = kTBar + 8;             // TMEM base address
  static constexpr uint32_t kSmemBytes = kSlot + 8;
  static constexpr uint32_t kTileBytesC = N * Q * 2, kTileBytesB = N * Q * 2,
                            kTileBytesX = P * Q * 2;
  // TMEM columns (fp32): G [0,128) then Yd [0,64); Yo [128,192); the state
  // [192, 192 + 64 NH) (rows n and n + 128 of lane n), which the state-update
  // product accumulates onto.
  static constexpr uint32_t kColG = 0, kColYd = 0, kColYo = 128, kColS = 192;
  static constexpr uint32_t kTmemCols = NH == 1 ? 256 : 512;
  static constexpr int kMinBlocks = NH == 1 ? 2 : 1;  // CTAs per SM
  static_assert(kMinBlocks * (kSmemBytes + 1024) <= 228 * 1024, "CTAs per SM (1 KB reserved each)");
  static_assert(kMinBlocks * kTmemCols <= 512, "TMEM columns per SM");
};
static_assert(Q == 128, "the masked block matrix shares the C / B tile layout");

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
// Shared-memory accesses at byte offsets from the dynamic base.
__device__ __forceinline__ void sts128(unsigned char* base, uint32_t off, const uint4& v) {
  *reinterpret_cast<uint4*>(base + off) = v;
}
__device__ __forceinline__ uint4 lds128(const unsigned char* base, uint32_t off) {
  return *reinterpret_cast<const uint4*>(base + off);
}
__device__ __forceinline__ uint4 ldg128(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
// Descriptor of a 128-byte-swizzled operand (layout type 2).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr, uint32_t k_stride, uint32_t mn_stride) {
  return umma::smem_desc(addr, k_stride, mn_stride) | (uint64_t(2) << 61);
}
// K-major swizzled operand with 128 rows, K in 64-column parts: the
// descriptor of K step k (16 elements): part k / 4, 32 bytes per step inside
// the 128-byte rows, 1024 bytes between 8-row groups.
__device__ __forceinline__ uint64_t desc_kmaj_sw(uint32_t tile, int k) {
  return desc_sw128(tile + (k >> 2) * kHalf + (k & 3) * 32, 16, 1024);
}
// MN-major swizzled operand (rows along K): K step k is 16 rows = 2048 bytes,
// 1024 bytes between 8-row groups, kHalf between 64-wide MN parts.
__device__ __forceinline__ uint64_t desc_mnmaj_sw(uint32_t tile, int k) {
  return desc_sw128(tile + k * 2048, kHalf, 1024);
}
__device__ __forceinline__ uint32_t swz(int row, int chunk) {  // byte offset in a swizzled part
  return row * 128 + ((chunk ^ (row & 7)) << 4);
}

// log2 with the MUFU unit (PTX lg2.approx.ftz.f32): -inf at 0.
__device__ __forceinline__ float lg2(float v) {
  float r;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

template <int NS, bool GATE>
__global__ void __launch_bounds__(2 * kThreads, SsdCfg<NS>::kMinBlocks)
    ssd_kernel(const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_b,
               const __grid_constant__ CUtensorMap tm_x, const SsdParams p) {
  using K = SsdCfg<NS>;
  constexpr int N = K::N, NQ = K::NQ, NH = K::NH;
  constexpr uint32_t kTileC = K::kTileC, kTileB = K::kTileB, kTileX = K::kTileX,
                     kTileXw = K::kTileXw, kTileS = K::kTileS, kStripS = K::kStripS;
  constexpr uint32_t kColG = K::kColG, kColYd = K::kColYd, kColYo = K::kColYo, kColS = K::kColS;
  extern __shared__ __align__(1024) unsigned char sm[];
  // 256 threads: thread (row, hf) handles row `row` of the block (step, or
  // state row) and the 32-column half `hf` of its 64 channels
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = tid & (kThreads - 1), hf = tid >> 7, lw = warp & 3;
  const int64_t H = p.nheads, L = p.seqlen, Dm = p.nheads * P;
  const int64_t b = blockIdx.x / H, h = blockIdx.x % H;
  const uint32_t s0 = umma::smem_u32(sm);
  const uint32_t bar = s0 + K::kBar, tbar = s0 + K::kTBar;
  float* sE = reinterpret_cast<float*>(sm + kTileXw);
  float* sF = sE + Q;
  float* sWt = reinterpret_cast<float*>(sm + K::kWarpTot);
  float* sD = reinterpret_cast<float*>(sm + K::kDs);
  const auto* dg = static_cast<const __nv_bfloat16*>(p.delta);
  const auto* zg = static_cast<const __nv_bfloat16*>(p.z);
  auto* yg = static_cast<__nv_bfloat16*>(p.y);

  int64_t Lv = L;
  if (p.valid_len) {
    Lv = p.valid_len[b];
    Lv = Lv < 0 ? 0 : (Lv > L ? L : Lv);
  }
  auto copy_c = [&](int64_t t0) {
    const int r = static_cast<int>(b * L + t0);
    umma::mbar_expect_tx(tbar, K::kTileBytesC);
#pragma unroll
    for (int q = 0; q < NQ; ++q) umma::tma_load_2d(s0 + kTileC + q * kHalf, &tm_c, 64 * q, r, tbar);
  };
  auto copy_bx = [&](int64_t t0) {
    const int r = static_cast<int>(b * L + t0);
    umma::mbar_expect_tx(tbar, K::kTileBytesB + K::kTileBytesX);
#pragma unroll
    for (int q = 0; q < NQ; ++q) umma::tma_load_2d(s0 + kTileB + q * kHalf, &tm_b, 64 * q, r, tbar);
    umma::tma_load_2d(s0 + kTileX, &tm_x, static_cast<int>(h * P), r, tbar);
  };
  if (s0 & 1023u) {
    if (tid == 0) atomicOr(p.err, kErrSsdAlign);
    return;
  }

  if (warp == 0) umma::tmem_alloc(s0 + K::kSlot, K::kTmemCols);
  if (tid == 0) {
    umma::mbar_init(bar, 2);
    umma::mbar_init(tbar, 2);
    if (Lv > 0) {
      copy_c(0);
      copy_bx(0);
    }
  }
  if (tid < P) sD[tid] = p.D ? __ldg(p.D + h * P + tid) : 0.f;
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tm = *reinterpret_cast<volatile uint32_t*>(sm + K::kSlot);
  const uint32_t tl = tm + (static_cast<uint32_t>(lw * 32) << 16);  // this warp's TMEM lanes
  const float al = __ldg(p.A + h) * kLog2e;
  const uint32_t rowo = row * 16;
  const int c0 = hf * 4;  // this thread's first 8-channel chunk

#pragma unroll
  for (int jh = 0; jh < NH; ++jh) {  // this thread's half of state row row + 128 jh: h0, else 0
    uint32_t r[32];
#pragma unroll
    for (int j = 0; j < 32; ++j)
      r[j] = __float_as_uint(
          p.h0 ? p.h0[((b * Dm + h * P + hf * 32 + j) * N) + row + 128 * jh] : 0.f);
    umma::tmem_st32(tl + kColS + 64 * jh + hf * 32, r);
  }
  umma::tmem_wait_st();

  uint32_t phase = 0, tphase = 0;
  int pending = Lv > 0 ? 2 : 0;
  int inflight = 0;
  bool bad = false;
  // The running sum of delta A over a block (log2 units) and the factors
  // derived from it, for row `row`: cs, e = cs - log2(delta), the column
  // factor toward the block's last step of the row's 32-step part, u =
  // delta 2^(cs_end - cs), and the block total.  A block's values are
  // computed while the previous block's second product runs.
  struct Scan {
    float cs, e, colf, u, tot;
  };
  auto scan_block = [&](float dt) {
    float cs = dt * al;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float v = __shfl_up_sync(0xFFFFFFFFu, cs, o);
      if (lane >= o) cs += v;
    }
    if (hf == 0 && lane == 31) sWt[lw] = cs;
    __syncthreads();
    float pre = 0.f, tot = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
      const float v = sWt[w];
      pre += w < lw ? v : 0.f;
      tot += v;
    }
    cs += pre;
    Scan r;
    r.cs = cs;
    r.e = cs - lg2(dt);
    r.colf = dt * ex2(__shfl_sync(0xFFFFFFFFu, cs, 31) - cs);
    r.u = dt * ex2(tot - cs);
    r.tot = tot;
    return r;
  };
  float dt_next = row < Lv ? __bfloat162float(dg[(b * L + row) * H + h]) : 0.f;
  Scan nxt = scan_block(dt_next);
  dt_next = row + Q < Lv ? __bfloat162float(dg[(b * L + row + Q) * H + h]) : 0.f;
  for (int64_t t0 = 0; t0 < L; t0 += Q) {
    const int64_t t = t0 + row;
    const bool in = t < Lv;
    const int64_t grow = b * L + t;
    if (t0 >= Lv) {
      if (t < L) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<uint4*>(yg + grow * Dm + h * P + (c0 + c) * 8) = make_uint4(0, 0, 0, 0);
      }
      continue;
    }
    const bool more = t0 + Q < Lv;
    const Scan cur = nxt;
    const float cs = cur.cs;

    {  // this thread's halves of the state rows: bf16 operand of Yo; kept scaled by
       // 2^cs_end (needs only the previous block's products, not this block's copies)
      const float etot = ex2(cur.tot);
#pragma unroll
      for (int jh = 0; jh < NH; ++jh) {
        uint32_t r0[32];
        umma::tmem_ld32_async(tl + kColS + 64 * jh + hf * 32, r0);
        umma::tmem_wait_ld(r0);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float f[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) f[j] = __uint_as_float(r0[c * 8 + j]);
          sts128(sm, kTileS + (c0 + c) * kStripS + (row + 128 * jh) * 16, pack8(f));
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) r0[j] = __float_as_uint(__uint_as_float(r0[j]) * etot);
        umma::tmem_st32(tl + kColS + 64 * jh + hf * 32, r0);
      }
      umma::tmem_wait_st();
    }

    if (umma::mbar_wait(tbar, tphase, kSsdWaitLimit)) {
      tphase ^= 1;
      pending = 0;
    } else {
      bad = true;
    }
    if (__syncthreads_or(bad)) { bad = true; break; }
    uint4 xr[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) xr[c] = in ? lds128(sm, kTileX + swz(row, c0 + c)) : make_uint4(0, 0, 0, 0);
    if (!in) {
#pragma unroll
      for (int q = hf; q < NQ; q += 2)
#pragma unroll
        for (int c = 0; c < 8; ++c)
          sts128(sm, kTileB + q * kHalf + row * 128 + c * 16, make_uint4(0, 0, 0, 0));
#pragma unroll
      for (int c = 0; c < 4; ++c) sts128(sm, kTileX + row * 128 + (c0 + c) * 16, make_uint4(0, 0, 0, 0));
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float f[8];
      unpack8(xr[c], f);
#pragma unroll
      for (int j = 0; j < 8; ++j) f[j] *= cur.u;
      sts128(sm, kTileXw + (c0 + c) * kStrip + rowo, pack8(f));
    }
    umma::fence_smem_to_async();
    umma::fence_before_sync();
    __syncthreads();

    if (tid == 0) {
      umma::fence_after_sync();
      constexpr uint32_t idG = umma::idesc_bf16(128, Q, false, false);
#pragma unroll
      for (int k = 0; k < N / 16; ++k)
        umma::mma_bf16(tm + kColG, desc_kmaj_sw(s0 + kTileC, k), desc_kmaj_sw(s0 + kTileB, k), idG,
                       k > 0);
      if (NH == 2) {  // the second half of the state rows (n >= 128), parts 2 and 3 of B
        constexpr uint32_t idS = umma::idesc_bf16(128, P, true, true);
#pragma unroll
        for (int k = 0; k < Q / 16; ++k)
          umma::mma_bf16(tm + kColS + 64, desc_mnmaj_sw(s0 + kTileB + 2 * kHalf, k),
                         umma::smem_desc(s0 + kTileXw + k * 256, 128, kStrip), idS, true);
      }
      umma::mma_commit(bar);
    }
    if (tid == 32) {
      umma::fence_after_sync();
      constexpr uint32_t idO = umma::idesc_bf16(128, P, false, true);
      constexpr uint32_t idS = umma::idesc_bf16(128, P, true, true);
#pragma unroll
      for (int k = 0; k < N / 16; ++k)
        umma::mma_bf16(tm + kColYo, desc_kmaj_sw(s0 + kTileC, k),
                       umma::smem_desc(s0 + kTileS + k * 256, 128, kStripS), idO, k > 0);
#pragma unroll
      for (int k = 0; k < Q / 16; ++k)
        umma::mma_bf16(tm + kColS, desc_mnmaj_sw(s0 + kTileB, k),
                       umma::smem_desc(s0 + kTileXw + k * 256, 128, kStrip), idS, true);
      umma::mma_commit(bar);
    }
    __syncwarp();
    inflight = 1;
    if (umma::mbar_wait(bar, phase, kSsdWaitLimit)) {
      phase ^= 1;
      --inflight;
    } else {
      bad = true;
    }
    if (__syncthreads_or(bad)) { bad = true; break; }
    umma::fence_after_sync();
    if (more) {
      pending = 1;
      if (tid == 0) copy_c(t0 + Q);
    }
    if (hf == 0) {
      sE[row] = cur.e;
      sF[row] = cur.colf;
    }
    __syncthreads();

    // Ym: parts sb = hf and hf + 2 of this row (32 columns each)
#pragma unroll
    for (int q2 = 0; q2 < 2; ++q2) {
      const int sb = hf + 2 * q2;
      uint4 o[4];
      if (sb <= lw) {  // warp-uniform
        uint32_t gr[32];
        umma::tmem_ld32_async(tl + kColG + sb * 32, gr);
        umma::tmem_wait_ld(gr);
        float g[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) g[j] = __uint_as_float(gr[j]);
        if (sb < lw) {
          float cref = 0.f;
#pragma unroll
          for (int w = 0; w < kThreads / 32; ++w) cref += w <= sb ? sWt[w] : 0.f;
          const float rf = ex2(cs - cref);
          const float4* f4 = reinterpret_cast<const float4*>(sF + sb * 32);
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const float4 f = f4[j4];
            g[j4 * 4 + 0] *= f.x * rf;
            g[j4 * 4 + 1] *= f.y * rf;
            g[j4 * 4 + 2] *= f.z * rf;
            g[j4 * 4 + 3] *= f.w * rf;
          }
        } else {
          const float4* e4 = reinterpret_cast<const float4*>(sE + sb * 32);
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const float4 ee = e4[j4];
            const float ev[4] = {ee.x, ee.y, ee.z, ee.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int j = j4 * 4 + i;
              g[j] = j <= lane ? g[j] * ex2(cs - ev[i]) : 0.f;
            }
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) o[q] = pack8(g + q * 8);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) o[q] = make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) sts128(sm, kTileB + (sb * 4 + q) * kStrip + rowo, o[q]);
    }
    uint4 zr[GATE ? 4 : 1];
    if (GATE) {
#pragma unroll
      for (int c = 0; c < 4; ++c)
        zr[c] = in ? ldg128(zg + grow * Dm + h * P + (c0 + c) * 8) : make_uint4(0, 0, 0, 0);
    }
    umma::fence_smem_to_async();
    umma::fence_before_sync();
    __syncthreads();

    if (tid == 0) {
      umma::fence_after_sync();
      constexpr uint32_t idY = umma::idesc_bf16(128, P, false, true);
#pragma unroll
      for (int k = 0; k < Q / 16; ++k)
        umma::mma_bf16(tm + kColYd, umma::smem_desc(s0 + kTileB + k * 2 * kStrip, kStrip, 128),
                       desc_mnmaj_sw(s0 + kTileX, k), idY, k > 0);
      umma::mma_commit(bar);
    }
    if (tid == 32) umma::mbar_arrive(bar);
    __syncwarp();
    inflight = 1;
    if (more) {  // the next block's running sums, while the product runs
      nxt = scan_block(dt_next);
      dt_next = t + 2 * Q < Lv ? __bfloat162float(dg[(grow + 2 * Q) * H + h]) : 0.f;
    }
    if (umma::mbar_wait(bar, phase, kSsdWaitLimit)) {
      phase ^= 1;
      --inflight;
    } else {
      bad = true;
    }
    if (__syncthreads_or(bad)) { bad = true; break; }
    umma::fence_after_sync();
    if (more) {
      pending = 2;
      if (tid == 0) copy_bx(t0 + Q);
    }

    // epilogue: y of step t = row, channels hf*32 .. hf*32 + 31
    const float eo = ex2(cs);
    {
      uint32_t yd[32], yo[32];
      umma::tmem_ld32_async(tl + kColYd + hf * 32, yd);
      umma::tmem_ld32_async(tl + kColYo + hf * 32, yo);
      umma::tmem_wait_ld(yd);
      umma::tmem_wait_ld(yo);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c = c0 + q;
        float xv[8], zv[8], o[8];
        unpack8(xr[q], xv);
        if (GATE) unpack8(zr[q], zv);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float v = fmaf(eo, __uint_as_float(yo[q * 8 + j]), __uint_as_float(yd[q * 8 + j]));
          v = fmaf(sD[c * 8 + j], xv[j], v);
          if (GATE) v *= silu(zv[j]);
          o[j] = in ? v : 0.f;
        }
        if (t < L) *reinterpret_cast<uint4*>(yg + grow * Dm + h * P + c * 8) = pack8(o);
      }
    }
    umma::fence_before_sync();
    __syncthreads();
  }

  if (bad) {
    if (tid == 0) atomicOr(p.err, kErrSsdWait);
    if (inflight > 0) umma::mbar_wait(bar, phase, kSsdWaitLimit);
  }
  if (pending > 0) {
    if (pending == 1 && tid == 0) umma::mbar_arrive(tbar);
    umma::mbar_wait(tbar, tphase, kSsdWaitLimit);
  }
  if (!bad && p.h_final) {
#pragma unroll
    for (int jh = 0; jh < NH; ++jh) {
      uint32_t r[32];
      umma::tmem_ld32_async(tl + kColS + 64 * jh + hf * 32, r);
      umma::tmem_wait_ld(r);
#pragma unroll
      for (int j = 0; j < 32; ++j)
        p.h_final[((b * Dm + h * P + hf * 32 + j) * N) + row + 128 * jh] = __uint_as_float(r[j]);
    }
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 0) umma::tmem_dealloc(tm, K::kTmemCols);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode() {
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

// 2-D map over a bf16 [rows, inner] tensor with a box of 64 elements x 128
// rows, 128-byte swizzled (one part of a tile).  Rows past the end read as zeros.
bool tile_map(CUtensorMap* m, const void* base, int64_t inner, int64_t rows) {
  EncodeTiledFn fn = encode();
  if (!fn) return false;
  cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(inner * 2)};
  cuuint32_t box[2] = {64, cuuint32_t(Q)};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NS, bool GATE>
cudaError_t launch_g(const CUtensorMap& mc, const CUtensorMap& mb, const CUtensorMap& mx,
                     const SsdParams& p, cudaStream_t s) {
  using K = SsdCfg<NS>;
  auto* k = ssd_kernel<NS, GATE>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(K::kSmemBytes));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  const int64_t grid = p.batch * p.nheads;
  k<<<static_cast<unsigned>(grid), 2 * kThreads, K::kSmemBytes, s>>>(mc, mb, mx, p);
  return cudaGetLastError();
}

}  // namespace

size_t ssd_smem_bytes(int64_t dstate) {
  return dstate == 256 ? SsdCfg<256>::kSmemBytes : SsdCfg<128>::kSmemBytes;
}

cudaError_t launch_ssd(const SsdParams& p, cudaStream_t s) {
  if (p.headdim != P || !ssd_supported_state(p.dstate) || p.batch * p.nheads <= 0 ||
      p.batch * p.nheads > 0x7FFFFFFF || p.batch * p.seqlen > 0x7FFFFFFF)
    return cudaErrorInvalidValue;
  CUtensorMap mc, mb, mx;
  const int64_t rows = p.batch * p.seqlen > 0 ? p.batch * p.seqlen : 1;
  if (!tile_map(&mc, p.C, p.dstate, rows) || !tile_map(&mb, p.B, p.dstate, rows) ||
      !tile_map(&mx, p.x, p.nheads * P, rows))
    return cudaErrorInvalidValue;
  if (p.dstate == 256)
    return p.z ? launch_g<256, true>(mc, mb, mx, p, s) : launch_g<256, false>(mc, mb, mx, p, s);
  return p.z ? launch_g<128, true>(mc, mb, mx, p, s) : launch_g<128, false>(mc, mb, mx, p, s);
}

}  // namespace ssm
