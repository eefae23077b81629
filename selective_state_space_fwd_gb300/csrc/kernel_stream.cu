// kernel_stream.cu -- host side of the STREAM tier: tensor maps, launch shape
// (states and channels per lane, warps per CTA, ring depth), eligibility and
// dispatch to the instances compiled in stream_inst_*.cu.  The kernel itself
// is in stream_core.cuh.
#include <cuda.h>

#include "stream_core.cuh"
#include "tiers.h"

namespace ssm {

// Sticky error word of the bounded waits (0 = no error).  Set with atomicOr
// by a CTA whose mbarrier wait gave up; read and cleared by the host through
// ssm_check_device_errors().
__device__ unsigned int g_stream_error = 0;

namespace stream {

SSM_STREAM_INSTANCES(SSM_STREAM_DECLARE)

unsigned int* error_word() {
  static unsigned int* addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (addr[dev] == nullptr) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_stream_error) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned int*>(a);
  }
  return addr[dev];
}

// Self-test of the bounded-wait error path.  One thread waits, with the same
// bounded wait as the kernels, on an mbarrier that nothing arrives on (no
// copy, no matrix product and no other thread targets it, so nothing is in
// flight when the kernel returns); after `polls` polls it gives up and sets
// the sticky error word exactly as a kernel whose copy never landed would.
__global__ void wait_timeout_selftest_kernel(unsigned polls, unsigned int* err) {
  __shared__ __align__(8) uint64_t bar;
  mbar_init(&bar, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if (!mbar_wait(&bar, 0, polls)) atomicOr(err, kErrWait);
}

// Dynamic shared memory a STREAM CTA may use (the opt-in limit of sm_103).
int max_dynamic_smem() { return 227 * 1024; }

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

bool tma_encode_available() { return encode_fn() != nullptr; }

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

namespace {

bool has_instance(int n, int g, int r) {
#define SSM_HAS(n_, g_, r_) \
  if (n == n_ && g == g_ && r == r_) return true;
  SSM_STREAM_INSTANCES(SSM_HAS)
#undef SSM_HAS
  return false;
}

int stage_bytes_of(int n, int g, int r, bool bf16, bool gate, int warps) {
#define SSM_SB(n_, g_, r_) \
  if (n == n_ && g == g_ && r == r_) return stage_bytes_ngr<n_, g_, r_>(bf16, gate, warps);
  SSM_STREAM_INSTANCES(SSM_SB)
#undef SSM_SB
  return 0;
}

}  // namespace

int sm_count() {
  static int count[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (count[dev] == 0) {
    int c = 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0)
      c = 148;
    count[dev] = c;
  }
  return count[dev];
}

namespace {

int channels_per_warp(int n, int g, int r) { return (32 / (n / g)) * r; }

// Bytes of a warp's partial-sum buffer.
int partial_bytes(int n, int g, int r) {
#define SSM_PB(n_, g_, r_) \
  if (n == n_ && g == g_ && r == r_) return Cfg<n_, g_, r_, float, false>::PBYTES;
  SSM_STREAM_INSTANCES(SSM_PB)
#undef SSM_PB
  return 0;
}

// Default (G, R): two channels per lane, four states (eight from 32 states
// up).  Measured on GB300 over the benchmark's workloads (8192 to 49152
// channels of 16 or 64 states): more (channel, state) pairs per lane cut the
// shared-memory traffic per pair but leave fewer warps to hide latency, and
// these problems have at most a few warps per scheduler to begin with.
void default_gr(const ScanParams& p, int* g, int* r) {
  *r = 2;
  switch (p.dstate) {
    case 4: case 8: case 16: *g = 4; break;
    case 32: case 64: *g = 8; break;
    default: *g = 0; *r = 0; break;
  }
}

}  // namespace
}  // namespace stream

StreamShape stream_shape(const ScanParams& p, bool bf16, int warps_per_block, int states_per_lane,
                         int channels_per_lane) {
  using namespace stream;
  StreamShape sh{0, 0, 0, 0};
  int g = states_per_lane, r = channels_per_lane;
  if (g == 0 || r == 0) {
    int dg = 0, dr = 0;
    default_gr(p, &dg, &dr);
    if (g == 0) g = dg;
    if (r == 0) r = dr;
  }
  if (g == 0 || r == 0 || !has_instance(p.dstate, g, r)) return sh;
  if (has_delta_prep(p) && !dtp_shape(p.dstate, g, r)) return sh;  // not compiled with it
  const int cw = channels_per_warp(p.dstate, g, r);
  const int sms = sm_count();
  const int64_t smem_sm = 228 * 1024;  // shared memory per SM
  // Ring depth for W warps per CTA: as many slots (2..4) as fit when every CTA
  // an SM is given is resident; 0 if not even two fit.
  auto stages_for = [&](int w, int64_t* per_sm_out) {
    const int sb = stage_bytes_of(p.dstate, g, r, bf16, p.z != nullptr, w);
    if (sb <= 0) return 0;
    const int64_t grid = (p.dim + int64_t(cw) * w - 1) / (int64_t(cw) * w) * p.batch;
    int64_t per_sm = (grid + sms - 1) / sms;
    const int64_t cap = 16 / w;  // about 16 warps per SM by registers
    if (per_sm > cap) per_sm = cap;
    *per_sm_out = per_sm;
    // per-warp partial-sum buffers (and fp32 delta slabs), barriers
    const int dsf = (bf16 && has_delta_prep(p)) ? 64 * cw * 4 : 0;
    const int fixed = w * (partial_bytes(p.dstate, g, r) + dsf) + 64;
    int st = static_cast<int>((smem_sm / per_sm - 1024 - fixed) / sb);
    if (st > 4) st = 4;
    if (st * sb + fixed > max_dynamic_smem()) st = (max_dynamic_smem() - fixed) / sb;
    return st >= 2 ? st : 0;
  };
  int w = warps_per_block, stages = 0;
  int64_t per_sm = 0;
  if (w != 0) {
    stages = stages_for(w, &per_sm);
    if (stages == 0) {  // the caller's W: two slots, even if not every CTA is resident
      const int sb = stage_bytes_of(p.dstate, g, r, bf16, p.z != nullptr, w);
      const int dsf = (bf16 && has_delta_prep(p)) ? 64 * cw * 4 : 0;
      if (sb <= 0 || 2 * sb + w * (partial_bytes(p.dstate, g, r) + dsf) + 64 > max_dynamic_smem())
        return sh;
      stages = 2;
    }
  } else {  // the fewest warps per CTA for which all CTAs are resident at once
    for (int c : {1, 2, 4}) {
      const int st = stages_for(c, &per_sm);
      if (st > 0) { w = c; stages = st; break; }
    }
    if (w == 0) {
      w = 4;
      stages = 2;
      const int sb = stage_bytes_of(p.dstate, g, r, bf16, p.z != nullptr, w);
      const int dsf = (bf16 && has_delta_prep(p)) ? 64 * cw * 4 : 0;
      if (sb <= 0 || 2 * sb + w * (partial_bytes(p.dstate, g, r) + dsf) + 64 > max_dynamic_smem())
        return sh;
    }
  }
  sh.wpc = w;
  sh.g = g;
  sh.r = r;
  sh.stages = stages;
  return sh;
}

cudaError_t launch_wait_timeout_selftest(unsigned polls, cudaStream_t s) {
  unsigned int* err = stream::error_word();
  if (err == nullptr) return cudaErrorInvalidValue;
  stream::wait_timeout_selftest_kernel<<<1, 1, 0, s>>>(polls, err);
  return cudaGetLastError();
}

bool read_and_clear_device_errors(unsigned int* word) {
  unsigned int zero = 0;
  if (cudaMemcpyFromSymbol(word, g_stream_error, sizeof(unsigned int)) != cudaSuccess) return false;
  return cudaMemcpyToSymbol(g_stream_error, &zero, sizeof(unsigned int)) == cudaSuccess;
}

bool stream_eligible(const ScanParams& p, bool bf16, StreamShape sh) {
  using namespace stream;
  if (sh.g == 0) return false;
  const int es = bf16 ? 2 : 4;
  const int cw = channels_per_warp(p.dstate, sh.g, sh.r);
  if (p.dstate * es < 16 || (cw * es) % 16 != 0) return false;
  if ((p.dim * es) % 16 != 0) return false;  // also makes dim a multiple of R
  if (p.seqlen > INT32_MAX || p.batch > INT32_MAX || p.dim > INT32_MAX / 2) return false;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(p.x) | reinterpret_cast<uintptr_t>(p.delta) |
                        reinterpret_cast<uintptr_t>(p.B) | reinterpret_cast<uintptr_t>(p.C) |
                        reinterpret_cast<uintptr_t>(p.z) | reinterpret_cast<uintptr_t>(p.y) |
                        reinterpret_cast<uintptr_t>(p.states) |
                        reinterpret_cast<uintptr_t>(p.h0) |
                        reinterpret_cast<uintptr_t>(p.h_final);
  if (mis % 16 != 0) return false;
  if (encode_fn() == nullptr) return false;
  return stream_grid(p, sh) <= INT32_MAX;
}

int64_t stream_grid(const ScanParams& p, StreamShape sh) {
  if (sh.g == 0) return 0;
  const int64_t cpc = int64_t(stream::channels_per_warp(p.dstate, sh.g, sh.r)) * sh.wpc;
  return (p.dim + cpc - 1) / cpc * p.batch;
}

namespace {

// The carry between segments of the time split, one thread per (b, d, n): the
// state entering segment s is the composition of the earlier segments'
// aggregates ([P1] s2.1: (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2)), segment
// s-1 contributing its decay product 2^(A log2(e) sum(delta)) and its end
// state from a zero start: h_s = P_{s-1} h_{s-1} + hend_{s-1}.
__global__ void seg_carry_kernel(const ScanParams p) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int N = p.dstate;
  if (i >= p.batch * p.dim * N) return;
  const int64_t n = i % N, d = (i / N) % p.dim, b = i / (int64_t(N) * p.dim);
  const float a = __ldg(p.A + d * N + n) * kLog2e;
  float* seg_h0 = const_cast<float*>(p.seg_h0);
  float h = p.seg_hend[((b * p.n_seg) * p.dim + d) * N + n];  // end of segment 0 (from h0)
  // The aggregates do not depend on the carried state: those of 16 segments
  // are loaded together, then composed in order.
  constexpr int CH = 16;
  for (int s0 = 1; s0 < p.n_seg; s0 += CH) {
    float dts[CH], he[CH];
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const int64_t row = b * p.n_seg + s0 + j;
      const bool need = s0 + j + 1 < p.n_seg;  // the last segment's aggregate is not used
      dts[j] = need ? p.seg_dtsum[row * p.dim + d] : 0.f;
      he[j] = need ? p.seg_hend[(row * p.dim + d) * N + n] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const int sg = s0 + j;
      if (sg < p.n_seg) {
        seg_h0[((b * p.n_seg + sg) * p.dim + d) * N + n] = h;
        h = fmaf(ex2(a * dts[j]), h, he[j]);
      }
    }
  }
}

}  // namespace

int64_t stream_auto_segments(const ScanParams& p, StreamShape sh) {
  // Split only when the rows leave most schedulers without a warp: then aim
  // at two warps per scheduler for 4 states per lane, four for 8 (twice the
  // dependent work per warp-step), with segments of at least 256 steps (the
  // aggregate pass costs about half a pass over all but the last segment).
  // Measured on GB300: b1 x L65536 x D256 x N16 (4 states per lane) is
  // fastest at two warps per scheduler (74 segments: 154 us; 147: 162 us);
  // b2 x L32768 x D512 x N64 (8 per lane) took 1127 us at two, 1014 us at
  // about four (20 segments) and 999 us at 32 segments.
  const int64_t warps = stream_grid(p, sh) * sh.wpc;
  const int64_t schedulers = 4 * int64_t(stream::sm_count());
  if (warps * 2 >= schedulers) return 1;
  const int64_t per_scheduler = sh.g >= 8 ? 4 : 2;
  int64_t segs = (per_scheduler * schedulers + warps - 1) / warps;
  const int64_t most = p.seqlen / 256;
  if (segs > most) segs = most;
  return segs < 1 ? 1 : segs;
}

cudaError_t launch_stream_agg(const ScanParams& p, bool bf16, cudaStream_t s, StreamShape sh) {
  using namespace stream;
#define SSM_GO_AGG(n_, g_, r_)                                \
  if (p.dstate == n_ && sh.g == g_ && sh.r == r_)             \
    return launch_ngr_agg<n_, g_, r_>(p, bf16, s, sh.wpc, sh.stages);
  SSM_STREAM_INSTANCES(SSM_GO_AGG)
#undef SSM_GO_AGG
  return cudaErrorInvalidValue;
}

cudaError_t launch_seg_carry(const ScanParams& p, cudaStream_t s) {
  const int64_t total = p.batch * p.dim * p.dstate;
  const int threads = 256;
  seg_carry_kernel<<<static_cast<unsigned>((total + threads - 1) / threads), threads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_stream(const ScanParams& p, bool bf16, cudaStream_t s, StreamShape sh) {
  using namespace stream;
#define SSM_GO(n_, g_, r_)                                   \
  if (p.dstate == n_ && sh.g == g_ && sh.r == r_)            \
    return launch_ngr<n_, g_, r_>(p, bf16, s, sh.wpc, sh.stages);
  SSM_STREAM_INSTANCES(SSM_GO)
#undef SSM_GO
  return cudaErrorInvalidValue;
}

}  // namespace ssm
