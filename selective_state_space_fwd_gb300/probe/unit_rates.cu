// unit_rates.cu -- throughput probes of the two arithmetic units the selective
// scan's roofline counts (libssmprobe.so; measurement harness, not part of
// the scan library).
//
//   ex2   : ex2.approx.ftz.f32 on the MUFU unit (one per decay exp(delta A))
//   ffma  : fma.rn.f32 on the fp32 pipe
//   ffma2 : fma.rn.f32x2 on the fp32 pipe (two lanes of work per instruction)
//   lds   : 16-byte shared-memory loads into registers, every lane its own
//           address (conflict-free), and the same with one address per warp
//           (a broadcast); the rate is bytes written to registers per clock,
//           the delivery that bounds kernels whose threads read their
//           operands from shared tiles
//
// One CTA of 1024 threads per SM (a large dynamic shared-memory request keeps
// a second CTA off the SM).  Every thread runs 8 independent dependency chains
// so that the unit, not latency, bounds the loop; each CTA times itself with
// clock64, so the result is in operations per SM clock, independent of the
// clock frequency.  The chains stay bounded: v <- 2^-v maps [1/2, 1] into
// itself, and v <- v * 0.999 + 0.001 converges to 1.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr int kThreads = 1024;
constexpr int kChains = 8;

__device__ __forceinline__ float ex2_neg(float v) {
  float r;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(-v));
  return r;
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1) rate_kernel(int iters, float seed,
                                                           long long* cycles, float* sink) {
  float v[kChains];
  unsigned long long w[kChains];
#pragma unroll
  for (int i = 0; i < kChains; ++i) {
    v[i] = 0.5f + 0.01f * ((threadIdx.x + i) & 31) * seed;
    const float lo = v[i], hi = v[i] * 0.5f;
    asm("mov.b64 %0, {%1, %2};" : "=l"(w[i]) : "f"(lo), "f"(hi));
  }
  const unsigned long long a2 = 0x3F7FBE773F7FBE77ull;  // {0.999f, 0.999f}
  const unsigned long long b2 = 0x3A83126F3A83126Full;  // {0.001f, 0.001f}
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < kChains; ++i) {
      if (KIND == 0) v[i] = ex2_neg(v[i]);
      if (KIND == 1) v[i] = fmaf(v[i], 0.999f, 0.001f);
      if (KIND == 2)
        asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(w[i]) : "l"(a2), "l"(b2));
    }
  }
  __syncthreads();
  const long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kChains; ++i) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(w[i]));
    s += v[i] + lo + hi;
  }
  if (s == 12345.678f) sink[threadIdx.x] = s;  // keeps the chains alive
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

// 16-byte shared-memory loads: kChains independent loads per iteration, each
// folded into an integer checksum.  The loads are ld.volatile (a plain load
// from an unchanged address could be hoisted out of the loop by the assembler,
// inline asm or not).  BCAST 0: lane l reads 16 bytes at 16 l of its chain's 512-byte
// row (each quarter warp covers the 32 banks once); BCAST 1: every lane of a
// warp reads the same 16 bytes.  Addresses stay inside 32 KB of the CTA's
// dynamic shared memory.
template <int BCAST>
__global__ void __launch_bounds__(kThreads, 1) lds_kernel(int iters, long long* cycles,
                                                          unsigned* sink) {
  extern __shared__ __align__(16) unsigned char sm[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < 32 * 1024 / 4; i += kThreads) reinterpret_cast<unsigned*>(sm)[i] = i;
  __syncthreads();
  const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(sm));
  uint32_t off[kChains];
#pragma unroll
  for (int i = 0; i < kChains; ++i)  // row (warp + 4 i) mod 64 of 512 bytes
    off[i] = base + ((warp + 4 * i) & 63) * 512 + (BCAST ? 0 : lane * 16);
  unsigned acc0 = 0, acc1 = 0;
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < kChains; ++i) {
      unsigned a, b, c, d;
      asm volatile("ld.volatile.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(off[i]));
      acc0 ^= a ^ b;
      acc1 ^= c ^ d;
    }
  }
  __syncthreads();
  const long long t1 = clock64();
  if ((acc0 ^ acc1) == 0x9e3779b9u) sink[tid] = acc0;  // keeps the loads' results live
  if (tid == 0) cycles[blockIdx.x] = t1 - t0;
}

// Lane l's byte offset, inside a 512-byte row, of the address patterns whose
// cost the scan kernels' lane layouts depend on (W = 16 or 8 bytes per lane):
//   0  every lane its own 16 bytes
//   1  one address for the warp (broadcast)
//   2  B/C slice of 4 states, state groups in consecutive lanes (l mod 4)
//   3  B/C slice of 4 states, the two lanes of a pair sharing a state group
//   4  first chunk of an 8-state B/C slice, consecutive lanes, rotated chunks
//   5  the same with pair-shared state groups
//   6  8-byte delta/x pair of 4-lane channel groups (l / 4)
//   7  8-byte delta/x pair of the pair-shared layout's channel groups
__device__ __forceinline__ uint32_t pattern_offset(int P, int l) {
  switch (P) {
    case 0: return l * 16;
    case 1: return 0;
    case 2: return (l & 3) * 16;
    case 3: return ((l >> 1) & 3) * 16;
    case 4: { const int sg = l & 7; return (2 * sg + ((sg >> 2) & 1)) * 16; }
    case 5: { const int sg = (l >> 1) & 7; return (2 * sg + ((sg >> 2) & 1)) * 16; }
    case 6: return (l >> 2) * 8;
    case 7: return (((l >> 3) << 1) | (l & 1)) * 8;
    default: return 0;
  }
}
constexpr int kPatterns = 8;

// Cycles per warp-wide load of pattern P (the shared-memory wavefronts it
// takes): kChains independent volatile loads per iteration, 16 bytes per lane
// for patterns 0-5 and 8 bytes for 6-7, rows inside 32 KB of the CTA's
// shared memory.
__global__ void __launch_bounds__(kThreads, 1) pattern_kernel(int P, int iters, long long* cycles,
                                                              unsigned* sink) {
  extern __shared__ __align__(16) unsigned char sm[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < 32 * 1024 / 4; i += kThreads) reinterpret_cast<unsigned*>(sm)[i] = i;
  __syncthreads();
  const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(sm));
  uint32_t off[kChains];
#pragma unroll
  for (int i = 0; i < kChains; ++i) off[i] = base + ((warp + 4 * i) & 63) * 512 + pattern_offset(P, lane);
  unsigned acc0 = 0, acc1 = 0;
  const long long t0 = clock64();
  if (P < 6) {
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int i = 0; i < kChains; ++i) {
        unsigned a, b, c, d;
        asm volatile("ld.volatile.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(off[i]));
        acc0 ^= a ^ b;
        acc1 ^= c ^ d;
      }
    }
  } else {
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int i = 0; i < kChains; ++i) {
        unsigned a, b;
        asm volatile("ld.volatile.shared.v2.u32 {%0, %1}, [%2];" : "=r"(a), "=r"(b) : "r"(off[i]));
        acc0 ^= a;
        acc1 ^= b;
      }
    }
  }
  __syncthreads();
  const long long t1 = clock64();
  if ((acc0 ^ acc1) == 0x9e3779b9u) sink[tid] = acc0;
  if (tid == 0) cycles[blockIdx.x] = t1 - t0;
}

// median over the SMs of the per-CTA cycle counts (sorts h in place)
double median_cycles(long long* h, int n) {
  for (int i = 1; i < n; ++i)
    for (int j = i; j > 0 && h[j - 1] > h[j]; --j) {
      const long long t = h[j];
      h[j] = h[j - 1];
      h[j - 1] = t;
    }
  return static_cast<double>(h[n / 2]);
}

template <int BCAST>
int run_lds(int sms, int iters, long long* d_cycles, unsigned* d_sink, double* out) {
  const int smem = 120 * 1024;  // one CTA per SM, as for the arithmetic probes
  if (cudaFuncSetAttribute(lds_kernel<BCAST>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return 1;
  lds_kernel<BCAST><<<sms, kThreads, smem>>>(iters, d_cycles, d_sink);  // warm-up
  lds_kernel<BCAST><<<sms, kThreads, smem>>>(iters, d_cycles, d_sink);
  if (cudaDeviceSynchronize() != cudaSuccess) return 2;
  long long* h = new long long[sms];
  if (cudaMemcpy(h, d_cycles, sizeof(long long) * sms, cudaMemcpyDeviceToHost) != cudaSuccess) {
    delete[] h;
    return 3;
  }
  const double cyc = median_cycles(h, sms);
  delete[] h;
  *out = double(kThreads) * kChains * iters * 16.0 / cyc;  // register bytes per clock
  return 0;
}

template <int KIND>
int run(int sms, int iters, long long* d_cycles, float* d_sink, double* out) {
  const int smem = 120 * 1024;  // more than half an SM's shared memory: one CTA per SM
  if (cudaFuncSetAttribute(rate_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return 1;
  rate_kernel<KIND><<<sms, kThreads, smem>>>(iters, 1.0f, d_cycles, d_sink);  // warm-up
  rate_kernel<KIND><<<sms, kThreads, smem>>>(iters, 1.0f, d_cycles, d_sink);
  if (cudaDeviceSynchronize() != cudaSuccess) return 2;
  long long* h = new long long[sms];
  if (cudaMemcpy(h, d_cycles, sizeof(long long) * sms, cudaMemcpyDeviceToHost) != cudaSuccess) {
    delete[] h;
    return 3;
  }
  // median over the SMs of lane-operations per clock
  const double cyc = median_cycles(h, sms);
  delete[] h;
  const double lanes_per_op = KIND == 2 ? 2.0 : 1.0;
  *out = double(kThreads) * kChains * iters * lanes_per_op / cyc;
  return 0;
}

}  // namespace

extern "C" {

// Measures, on the current device, MUFU ex2 results per SM clock and fp32 FMA
// lane-operations per SM clock (scalar and f32x2 forms).  Returns 0 on
// success; *sms receives the SM count.
int ssmprobe_unit_rates(double* ex2_per_clk, double* ffma_per_clk, double* ffma2_per_clk,
                        int* sms) {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 10;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 11;
  *sms = n;
  long long* d_cycles = nullptr;
  float* d_sink = nullptr;
  if (cudaMalloc(&d_cycles, sizeof(long long) * n) != cudaSuccess) return 12;
  if (cudaMalloc(&d_sink, sizeof(float) * kThreads) != cudaSuccess) {
    cudaFree(d_cycles);
    return 12;
  }
  int rc = run<0>(n, 4096, d_cycles, d_sink, ex2_per_clk);
  if (rc == 0) rc = run<1>(n, 8192, d_cycles, d_sink, ffma_per_clk);
  if (rc == 0) rc = run<2>(n, 4096, d_cycles, d_sink, ffma2_per_clk);
  cudaFree(d_cycles);
  cudaFree(d_sink);
  return rc;
}

// Measures, on the current device, the cycles per warp-wide shared-memory
// load of each address pattern of pattern_offset (out[kPatterns]).  Returns
// 0 on success.
int ssmprobe_lds_patterns(double* cycles_per_load, int n) {
  if (n < kPatterns) return 13;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 10;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return 11;
  long long* d_cycles = nullptr;
  unsigned* d_sink = nullptr;
  if (cudaMalloc(&d_cycles, sizeof(long long) * sms) != cudaSuccess) return 12;
  if (cudaMalloc(&d_sink, sizeof(unsigned) * kThreads) != cudaSuccess) {
    cudaFree(d_cycles);
    return 12;
  }
  const int smem = 120 * 1024, iters = 1024;
  int rc = cudaFuncSetAttribute(pattern_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ==
                   cudaSuccess ? 0 : 1;
  long long* h = new long long[sms];
  for (int P = 0; P < kPatterns && rc == 0; ++P) {
    pattern_kernel<<<sms, kThreads, smem>>>(P, iters, d_cycles, d_sink);  // warm-up
    pattern_kernel<<<sms, kThreads, smem>>>(P, iters, d_cycles, d_sink);
    if (cudaDeviceSynchronize() != cudaSuccess) { rc = 2; break; }
    if (cudaMemcpy(h, d_cycles, sizeof(long long) * sms, cudaMemcpyDeviceToHost) != cudaSuccess) {
      rc = 3;
      break;
    }
    const double warp_loads = double(kThreads / 32) * kChains * iters;
    cycles_per_load[P] = median_cycles(h, sms) / warp_loads;
  }
  delete[] h;
  cudaFree(d_cycles);
  cudaFree(d_sink);
  return rc;
}

// Measures, on the current device, the bytes per SM clock that 16-byte
// shared-memory loads write into registers: every lane its own address
// (conflict-free) and one address per warp (broadcast).  Returns 0 on success.
int ssmprobe_lds_rates(double* bytes_per_clk, double* bcast_bytes_per_clk) {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 10;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 11;
  long long* d_cycles = nullptr;
  unsigned* d_sink = nullptr;
  if (cudaMalloc(&d_cycles, sizeof(long long) * n) != cudaSuccess) return 12;
  if (cudaMalloc(&d_sink, sizeof(unsigned) * kThreads) != cudaSuccess) {
    cudaFree(d_cycles);
    return 12;
  }
  int rc = run_lds<0>(n, 2048, d_cycles, d_sink, bytes_per_clk);
  if (rc == 0) rc = run_lds<1>(n, 2048, d_cycles, d_sink, bcast_bytes_per_clk);
  cudaFree(d_cycles);
  cudaFree(d_sink);
  return rc;
}

}  // extern "C"
