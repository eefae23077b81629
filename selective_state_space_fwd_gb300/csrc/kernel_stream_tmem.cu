// kernel_stream_tmem.cu -- host side of the STREAM-TM tier (stream_tmem.cuh):
// tensor maps, shared-memory ring depth, eligibility and the launch.  The
// instances are compiled in stream_tmem_inst_n*.cu.
#include <cuda.h>

#include "stream_tmem.cuh"
#include "tiers.h"

namespace ssm {
namespace stream_tm {

// Instances: (dstate, states per lane, channels per lane, compute warps per
// CTA).  Defined in stream_tmem_inst_n*.cu.
template <int N, int G, int R, int W>
cudaError_t launch_ngw(const ScanParams& p, bool bf16, cudaStream_t s, int stages);
template <int N, int G, int R, int W>
int smem_ngw(bool bf16, bool gate, int stages);

#define SSM_TM_INSTANCES(X) X(16, 4, 1, 8) X(16, 4, 2, 4) X(64, 8, 1, 8) X(64, 8, 2, 4)
#define SSM_TM_DECLARE(N_, G_, R_, W_)                                                       \
  template <>                                                                                \
  cudaError_t launch_ngw<N_, G_, R_, W_>(const ScanParams&, bool, cudaStream_t, int);        \
  template <>                                                                                \
  int smem_ngw<N_, G_, R_, W_>(bool, bool, int);
SSM_TM_INSTANCES(SSM_TM_DECLARE)

namespace {
int states_per_lane(int n) { return n <= 16 ? 4 : 8; }
// compute warps per CTA: one CTA per SM holds all of its TMEM, so the CTA
// carries as many warps as the lane layout leaves per SM on the benchmark's
// workloads (one channel per lane: twice the lanes)
int warps_for(int r) { return r == 1 ? 8 : 4; }
constexpr int kMaxSmem = 227 * 1024;
}  // namespace

}  // namespace stream_tm

StreamTmShape stream_tm_shape(const ScanParams& p, bool bf16, int channels_per_lane) {
  using namespace stream_tm;
  StreamTmShape sh{0, 0, 0, 0};
  const int g = states_per_lane(p.dstate);
  const int r = channels_per_lane == 0 ? 2 : channels_per_lane;
  const int w = warps_for(r);
  int (*smem)(bool, bool, int) = nullptr;
#define SSM_TM_SMEM(N_, G_, R_, W_) \
  if (p.dstate == N_ && g == G_ && r == R_ && w == W_) smem = smem_ngw<N_, G_, R_, W_>;
  SSM_TM_INSTANCES(SSM_TM_SMEM)
#undef SSM_TM_SMEM
  if (smem == nullptr) return sh;
  int stages = 0;
  for (int st = 4; st >= 2; --st)
    if (smem(bf16, p.z != nullptr, st) > 0 && smem(bf16, p.z != nullptr, st) <= kMaxSmem) {
      stages = st;
      break;
    }
  if (stages == 0) return sh;
  sh.g = g;
  sh.r = r;
  sh.warps = w;
  sh.stages = stages;
  return sh;
}

bool stream_tm_eligible(const ScanParams& p, bool bf16, StreamTmShape sh) {
  if (sh.g == 0) return false;
  if (has_delta_prep(p)) return false;  // the fused step-size preparation runs in STREAM
  const int es = bf16 ? 2 : 4;
  const int cw = 32 / (p.dstate / sh.g) * sh.r;
  if ((cw * es) % 16 != 0 || (p.dstate * es) % 16 != 0) return false;
  if ((p.dim * es) % 16 != 0) return false;
  if (p.seqlen > INT32_MAX || p.batch > INT32_MAX || p.dim > INT32_MAX / 2) return false;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(p.x) | reinterpret_cast<uintptr_t>(p.delta) |
                        reinterpret_cast<uintptr_t>(p.B) | reinterpret_cast<uintptr_t>(p.C) |
                        reinterpret_cast<uintptr_t>(p.z) | reinterpret_cast<uintptr_t>(p.y) |
                        reinterpret_cast<uintptr_t>(p.states) |
                        reinterpret_cast<uintptr_t>(p.h0) |
                        reinterpret_cast<uintptr_t>(p.h_final);
  if (mis % 16 != 0) return false;
  return stream_tm_grid(p, sh) <= INT32_MAX;
}

int64_t stream_tm_grid(const ScanParams& p, StreamTmShape sh) {
  if (sh.g == 0) return 0;
  const int64_t cpc = int64_t(32 / (p.dstate / sh.g)) * sh.r * sh.warps;
  return (p.dim + cpc - 1) / cpc * p.batch;
}

cudaError_t launch_stream_tm(const ScanParams& p, bool bf16, cudaStream_t s, StreamTmShape sh) {
  using namespace stream_tm;
#define SSM_TM_GO(N_, G_, R_, W_)                                           \
  if (p.dstate == N_ && sh.g == G_ && sh.r == R_ && sh.warps == W_)         \
    return launch_ngw<N_, G_, R_, W_>(p, bf16, s, sh.stages);
  SSM_TM_INSTANCES(SSM_TM_GO)
#undef SSM_TM_GO
  return cudaErrorInvalidValue;
}

}  // namespace ssm
