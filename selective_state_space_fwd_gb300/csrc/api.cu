// api.cu -- the C ABI of libssmscan (declared in include/ssmscan.h).
//
// Host-side only: argument validation, choice of kernel tier, launch.  Every
// argument error is found here, before anything is enqueued, and is returned
// as an ssm_status; nothing aborts or throws across the ABI.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <new>

#include "ssmscan.h"
#include "ssd.h"
#include "tiers.h"

namespace {

using ssm::ScanParams;

constexpr int64_t kBwdMaxChunk = 512;  // longest chunk the backward replays in shared memory
constexpr uint32_t kSelftestMaxPolls = 1u << 20;  // bound of ssm_selftest_wait_timeout

bool supported_dstate(int64_t n) {
  return n == 1 || n == 2 || n == 4 || n == 8 || n == 16 || n == 32 || n == 64;
}

size_t elem_size(ssm_dtype t) { return t == SSM_BF16 ? 2 : 4; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// a * b without signed overflow, for non-negative operands; false on overflow.
bool mul_ok(int64_t a, int64_t b, int64_t* out) {
  if (a != 0 && b > INT64_MAX / a) return false;
  *out = a * b;
  return true;
}

// Shape checks shared by every entry point.  Element counts are kept below
// 2^60 so that byte offsets of every tensor fit in int64.
ssm_status check_shapes(const ssm_shapes* s, ssm_dtype dtype, bool want_states) {
  if (s == nullptr) return SSM_ERR_NULL;
  if (dtype != SSM_F32 && dtype != SSM_BF16) return SSM_ERR_UNSUPPORTED;
  if (s->batch < 1 || s->seqlen < 1 || s->dim < 1 || s->dstate < 1) return SSM_ERR_SHAPE;
  if (!supported_dstate(s->dstate)) return SSM_ERR_UNSUPPORTED;
  if (s->chunk_len < 0) return SSM_ERR_SHAPE;
  if (want_states && s->chunk_len == 0) return SSM_ERR_SHAPE;
  int64_t bl, bld, bln, dn;
  const int64_t lim = int64_t(1) << 60;
  if (!mul_ok(s->batch, s->seqlen, &bl) || !mul_ok(bl, s->dim, &bld) ||
      !mul_ok(bl, s->dstate, &bln) || !mul_ok(s->dim, s->dstate, &dn))
    return SSM_ERR_SHAPE;
  if (bld > lim || bln > lim || dn > lim) return SSM_ERR_SHAPE;
  if (want_states) {
    int64_t st;
    const int64_t nch = (s->seqlen + s->chunk_len - 1) / s->chunk_len;
    if (!mul_ok(s->batch, nch, &st) || !mul_ok(st, dn, &st) || st > lim) return SSM_ERR_SHAPE;
  }
  return SSM_OK;
}

ssm_status check_options(const ssm_options* o) {
  if (o == nullptr) return SSM_OK;
  if (o->warps_per_block != 0 && o->warps_per_block != 1 && o->warps_per_block != 2 &&
      o->warps_per_block != 4)
    return SSM_ERR_UNSUPPORTED;
  if (o->kernel < SSM_KERNEL_AUTO || o->kernel > SSM_KERNEL_STREAM_TM) return SSM_ERR_UNSUPPORTED;
  if (o->states_per_lane != 0 && o->states_per_lane != 2 && o->states_per_lane != 4 &&
      o->states_per_lane != 8 && o->states_per_lane != 16)
    return SSM_ERR_UNSUPPORTED;
  if (o->channels_per_lane != 0 && o->channels_per_lane != 2 && o->channels_per_lane != 4 &&
      !(o->channels_per_lane == 1 && o->kernel == SSM_KERNEL_STREAM_TM))
    return SSM_ERR_UNSUPPORTED;
  return SSM_OK;
}

struct Plan {
  ssm_kernel kernel;
  int64_t grid;
  ssm::StreamShape shape;
  ssm::StreamTmShape tm_shape;
};

// Tier choice.  `forced` is the caller's request (AUTO = let the library pick).
ssm_status make_plan(const ScanParams& p, ssm_dtype dtype, const ssm_options* o, Plan* out) {
  const bool bf16 = dtype == SSM_BF16;
  const ssm_kernel forced = o ? o->kernel : SSM_KERNEL_AUTO;
  const ssm::StreamShape shape =
      ssm::stream_shape(p, bf16, o ? o->warps_per_block : 0, o ? o->states_per_lane : 0,
                        o ? o->channels_per_lane : 0);
  ssm_kernel k = forced;
  if (k == SSM_KERNEL_AUTO)
    k = ssm::stream_eligible(p, bf16, shape) ? SSM_KERNEL_STREAM : SSM_KERNEL_SERIAL;
  out->kernel = k;
  out->shape = shape;
  out->tm_shape = ssm::StreamTmShape{0, 0, 0, 0};
  switch (k) {
    case SSM_KERNEL_SERIAL:
      out->grid = ssm::serial_grid(p);
      return SSM_OK;
    case SSM_KERNEL_STREAM:
      if (!ssm::stream_eligible(p, bf16, shape)) return SSM_ERR_UNSUPPORTED;
      out->grid = ssm::stream_grid(p, shape);
      return SSM_OK;
    case SSM_KERNEL_WARPSCAN:
      if (!ssm::warpscan_eligible(p)) return SSM_ERR_UNSUPPORTED;
      out->grid = ssm::warpscan_grid(p);
      return SSM_OK;
    case SSM_KERNEL_STREAM_TM: {
      // the tier's launch shape follows from dstate and the lane layout
      if (o && (o->warps_per_block || o->states_per_lane || o->channels_per_lane > 2))
        return SSM_ERR_UNSUPPORTED;
      const ssm::StreamTmShape tm = ssm::stream_tm_shape(p, bf16, o ? o->channels_per_lane : 0);
      if (!ssm::stream_tm_eligible(p, bf16, tm)) return SSM_ERR_UNSUPPORTED;
      out->tm_shape = tm;
      out->grid = ssm::stream_tm_grid(p, tm);
      return SSM_OK;
    }
    default:
      return SSM_ERR_UNSUPPORTED;
  }
}

ScanParams make_params(const void* x, const void* delta, const float* A, const void* B,
                       const void* C, const float* D, const void* z, const int32_t* valid_len,
                       void* y, float* states, const ssm_shapes* s, const float* h0 = nullptr,
                       float* h_final = nullptr) {
  ScanParams p;
  p.x = x; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z;
  p.valid_len = valid_len; p.y = y; p.h0 = h0; p.h_final = h_final;
  p.batch = s->batch; p.seqlen = s->seqlen; p.dim = s->dim;
  p.dstate = static_cast<int>(s->dstate);
  const bool st = states != nullptr && s->chunk_len > 0;
  p.states = st ? states : nullptr;
  p.chunk_len = st ? s->chunk_len : 1;
  p.n_chunks = st ? (s->seqlen + s->chunk_len - 1) / s->chunk_len : 0;
  p.len_offset = 0;
  p.dt_bias = nullptr;
  p.delta_softplus = 0;
  p.delta_clamp = 0;
  p.delta_lo = 0.f;
  p.delta_hi = 0.f;
  p.seg_len = 0;
  p.n_seg = 1;
  p.seg_h0 = nullptr;
  p.seg_hend = nullptr;
  p.seg_dtsum = nullptr;
  return p;
}

// Validates and applies the fused step-size preparation to the kernel parameters.
template <class P>
ssm_status apply_prep(const ssm_delta_prep* prep, P* p) {
  if (prep == nullptr) return SSM_OK;
  if (prep->dt_bias && !aligned(prep->dt_bias, 4)) return SSM_ERR_ALIGN;
  if ((prep->softplus != 0 && prep->softplus != 1) || (prep->clamp != 0 && prep->clamp != 1))
    return SSM_ERR_UNSUPPORTED;
  if (prep->clamp && !(prep->lo <= prep->hi)) return SSM_ERR_SHAPE;  // also rejects NaN
  p->dt_bias = prep->dt_bias;
  p->delta_softplus = prep->softplus;
  p->delta_clamp = prep->clamp;
  p->delta_lo = prep->lo;
  p->delta_hi = prep->hi;
  return SSM_OK;
}

// The entry points keep per-device state (the sticky error word of the
// bounded waits, copy streams, the address of the fixed workspace) and look it
// up by the calling thread's current device; `stream` must belong to that
// device, else SSM_ERR_CUDA.  The special handles (0, legacy, per-thread)
// always do.
ssm_status current_device_for(cudaStream_t stream, int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) return SSM_ERR_CUDA;
  if (stream == nullptr || stream == cudaStreamLegacy || stream == cudaStreamPerThread)
    return SSM_OK;
  // A stream being captured into a CUDA graph is not queried for its device
  // (the query would invalidate the capture); the calls then only record work.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return SSM_ERR_CUDA;
  if (cap != cudaStreamCaptureStatusNone) return SSM_OK;
  int sdev = -1;
  if (cudaStreamGetDevice(stream, &sdev) != cudaSuccess) return SSM_ERR_CUDA;
  return sdev == *dev ? SSM_OK : SSM_ERR_CUDA;
}

// Launch the planned tier.
ssm_status launch(const ScanParams& p, ssm_dtype dtype, const ssm_options* opts,
                  cudaStream_t stream) {
  Plan plan;
  ssm_status st = make_plan(p, dtype, opts, &plan);
  if (st != SSM_OK) return st;
  int dev = 0;
  if ((st = current_device_for(stream, &dev)) != SSM_OK) return st;
  const bool bf16 = dtype == SSM_BF16;
  cudaError_t err = cudaErrorInvalidValue;
  switch (plan.kernel) {
    case SSM_KERNEL_SERIAL: err = ssm::launch_serial(p, bf16, stream); break;
    case SSM_KERNEL_STREAM: err = ssm::launch_stream(p, bf16, stream, plan.shape); break;
    case SSM_KERNEL_WARPSCAN: err = ssm::launch_warpscan(p, bf16, stream); break;
    case SSM_KERNEL_STREAM_TM: err = ssm::launch_stream_tm(p, bf16, stream, plan.tm_shape); break;
    default: return SSM_ERR_UNSUPPORTED;
  }
  return err == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Byte layout of the device workspace used by ssm_scan_fwd_host.  `total` is
// SIZE_MAX when a region size or the running sum would not fit in size_t.
struct HostLayout {
  size_t x, delta, z, B, C, A, D, valid, y, states, carry, total;
};

constexpr size_t kNoFit = SIZE_MAX;

// a * b, or kNoFit when it does not fit.
size_t mul_size(size_t a, size_t b) {
  if (a != 0 && b > (kNoFit - 1) / a) return kNoFit;
  return a * b;
}

HostLayout host_layout(const ssm_shapes* s, ssm_dtype dtype, int has_D, int has_z, int has_valid,
                       int has_states) {
  const size_t es = elem_size(dtype);
  const size_t bl = mul_size(size_t(s->batch), size_t(s->seqlen));
  const size_t act = mul_size(mul_size(bl, size_t(s->dim)), es);
  const size_t bc = mul_size(mul_size(bl, size_t(s->dstate)), es);
  const size_t dn4 = mul_size(mul_size(size_t(s->dim), size_t(s->dstate)), 4);
  const size_t nch = s->chunk_len > 0 ? size_t((s->seqlen + s->chunk_len - 1) / s->chunk_len) : 0;
  HostLayout l;
  size_t off = 0;
  bool fits = true;
  // region of `bytes` at the current offset; the next starts 256-byte aligned
  auto take = [&](size_t bytes) {
    const size_t o = off;
    if (bytes > kNoFit - 256 || off > kNoFit - 256 - bytes) {
      fits = false;
      return size_t(0);
    }
    off = round_up(off + bytes, 256);
    return o;
  };
  l.x = take(act);
  l.delta = take(act);
  l.z = has_z ? take(act) : 0;
  l.B = take(bc);
  l.C = take(bc);
  l.A = take(dn4);
  l.D = has_D ? take(mul_size(size_t(s->dim), 4)) : 0;
  l.valid = has_valid ? take(mul_size(size_t(s->batch), 4)) : 0;
  l.y = take(act);
  l.states = has_states ? take(mul_size(mul_size(size_t(s->batch), nch), dn4)) : 0;
  l.carry = take(mul_size(2 * size_t(s->batch), dn4));
  l.total = fits ? off : kNoFit;
  return l;
}

// ---- the end-to-end form: copies and kernels pipelined over time pieces ----------
//
// The sequence is cut into pieces of `piece` steps.  Piece i's inputs are
// copied host -> device on a copy stream, its kernel runs on the caller's
// stream starting from the state piece i-1 ended in (the serial carry between
// sequence chunks, [P1] s3.1 third level, [P2] s2.4), and its outputs are
// copied device -> host on a second copy stream, so that the two copy
// directions and the kernels of neighbouring pieces overlap.  In the workspace
// every tensor is stored piece-major (piece i holds [batch, piece, ...]
// contiguous), so each kernel sees an ordinary compact problem and each copy is
// one strided 2-D copy.

#ifndef SSM_HOST_PIECES
#define SSM_HOST_PIECES 8  // pieces per call when the sequence is long enough
#endif

// Library-owned copy streams and the events that chain them, one set per device.
struct HostStreams {
  std::mutex mu;        // one call enqueues on a device's set at a time
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, in = nullptr, kern = nullptr, done = nullptr;
};

constexpr int kMaxDevices = 64;
HostStreams g_host_streams[kMaxDevices];
std::mutex g_host_streams_mu;

HostStreams* host_streams(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  HostStreams* h = &g_host_streams[dev];
  std::lock_guard<std::mutex> lk(g_host_streams_mu);
  if (!h->ready) {
    const unsigned ef = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&h->h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&h->d2h, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->start, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->in, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->kern, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->done, ef) != cudaSuccess)
      return nullptr;
    h->ready = true;
  }
  return h;
}

// Steps per piece: about SSM_HOST_PIECES pieces, a multiple of 64 steps (the
// STREAM tile), a multiple of chunk_len when chunk states are wanted (so that
// every chunk lies inside one piece), and at least 1 MiB of input per piece.
int64_t host_piece_steps(const ssm_shapes& s, ssm_dtype dtype, bool has_z, bool want_states) {
  const int64_t L = s.seqlen;
  const int64_t es = static_cast<int64_t>(elem_size(dtype));
  const int64_t step_bytes = s.batch * es * ((has_z ? 3 : 2) * s.dim + 2 * s.dstate);
  int64_t piece = (L + SSM_HOST_PIECES - 1) / SSM_HOST_PIECES;
  const int64_t min_steps = ((int64_t(1) << 20) + step_bytes - 1) / step_bytes;
  if (piece < min_steps) piece = min_steps;
  piece = (piece + 63) / 64 * 64;
  if (want_states) piece = (piece + s.chunk_len - 1) / s.chunk_len * s.chunk_len;
  return piece < L ? piece : L;
}

ssm_status run_host_pipeline(const void* x, const void* delta, const float* A, const void* B,
                             const void* C, const float* D, const void* z,
                             const int32_t* valid_len, void* out_y, float* out_states,
                             const ssm_shapes& s, ssm_dtype dtype, char* ws, const HostLayout& l,
                             cudaStream_t stream) {
  int dev = 0;
  const ssm_status ds = current_device_for(stream, &dev);
  if (ds != SSM_OK) return ds;
  HostStreams* hs = host_streams(dev);
  if (hs == nullptr) return SSM_ERR_CUDA;
  std::lock_guard<std::mutex> lk(hs->mu);

  const bool want_states = out_states != nullptr;
  const size_t es = elem_size(dtype);
  const int64_t L = s.seqlen, Bt = s.batch, N = s.dstate;
  const size_t dn4 = size_t(s.dim) * N * 4;
  const int64_t nch = want_states ? (L + s.chunk_len - 1) / s.chunk_len : 0;
  const int64_t piece = host_piece_steps(s, dtype, z != nullptr, want_states);
  float* carry[2] = {reinterpret_cast<float*>(ws + l.carry),
                     reinterpret_cast<float*>(ws + l.carry + size_t(Bt) * dn4)};

  cudaError_t e = cudaSuccess;
  auto ok = [&](cudaError_t r) { if (e == cudaSuccess) e = r; return e == cudaSuccess; };
  // [batch, L, w] host tensor, steps [t0, t0 + n) -> piece-major workspace region
  auto copy_in = [&](size_t region, const void* src, int64_t w, int64_t t0, int64_t n) {
    const size_t row = size_t(w) * es;
    return ok(cudaMemcpy2DAsync(ws + region + size_t(Bt) * t0 * row, n * row,
                                static_cast<const char*>(src) + t0 * row, L * row, n * row, Bt,
                                cudaMemcpyHostToDevice, hs->h2d));
  };

  // the caller's earlier work on `stream` (e.g. on this workspace) comes first
  ok(cudaEventRecord(hs->start, stream));
  ok(cudaStreamWaitEvent(hs->h2d, hs->start, 0));
  ok(cudaStreamWaitEvent(hs->d2h, hs->start, 0));
  ok(cudaMemcpyAsync(ws + l.A, A, dn4, cudaMemcpyHostToDevice, hs->h2d));
  if (D) ok(cudaMemcpyAsync(ws + l.D, D, size_t(s.dim) * 4, cudaMemcpyHostToDevice, hs->h2d));
  if (valid_len)
    ok(cudaMemcpyAsync(ws + l.valid, valid_len, size_t(Bt) * 4, cudaMemcpyHostToDevice, hs->h2d));

  ssm_status st = SSM_OK;
  int i = 0;
  for (int64_t t0 = 0; t0 < L && e == cudaSuccess && st == SSM_OK; t0 += piece, ++i) {
    const int64_t n = L - t0 < piece ? L - t0 : piece;
    const size_t act_off = size_t(Bt) * t0 * s.dim * es, bc_off = size_t(Bt) * t0 * N * es;
    copy_in(l.x, x, s.dim, t0, n);
    copy_in(l.delta, delta, s.dim, t0, n);
    if (z) copy_in(l.z, z, s.dim, t0, n);
    copy_in(l.B, B, N, t0, n);
    copy_in(l.C, C, N, t0, n);
    ok(cudaEventRecord(hs->in, hs->h2d));
    ok(cudaStreamWaitEvent(stream, hs->in, 0));
    if (e != cudaSuccess) break;

    const int64_t c0 = want_states ? t0 / s.chunk_len : 0;
    const int64_t pch = want_states ? (n + s.chunk_len - 1) / s.chunk_len : 0;
    float* pstates = want_states ? reinterpret_cast<float*>(ws + l.states) + size_t(Bt) * c0 *
                                       (dn4 / 4)
                                 : nullptr;
    const ssm_shapes ps = {Bt, n, s.dim, N, want_states ? s.chunk_len : 0};
    ScanParams p = make_params(ws + l.x + act_off, ws + l.delta + act_off,
                               reinterpret_cast<const float*>(ws + l.A), ws + l.B + bc_off,
                               ws + l.C + bc_off,
                               D ? reinterpret_cast<const float*>(ws + l.D) : nullptr,
                               z ? ws + l.z + act_off : nullptr,
                               valid_len ? reinterpret_cast<const int32_t*>(ws + l.valid) : nullptr,
                               ws + l.y + act_off, pstates, &ps,
                               t0 == 0 ? nullptr : carry[i % 2],
                               t0 + n < L ? carry[(i + 1) % 2] : nullptr);
    p.len_offset = t0;
    st = launch(p, dtype, nullptr, stream);
    if (st != SSM_OK) break;
    ok(cudaEventRecord(hs->kern, stream));
    ok(cudaStreamWaitEvent(hs->d2h, hs->kern, 0));
    const size_t row = size_t(s.dim) * es;
    ok(cudaMemcpy2DAsync(static_cast<char*>(out_y) + t0 * row, L * row, ws + l.y + act_off,
                         n * row, n * row, Bt, cudaMemcpyDeviceToHost, hs->d2h));
    if (want_states)
      ok(cudaMemcpy2DAsync(out_states + size_t(c0) * (dn4 / 4), nch * dn4, pstates, pch * dn4,
                           pch * dn4, Bt, cudaMemcpyDeviceToHost, hs->d2h));
  }
  // join: the caller's stream reaches the end only after the last copy out
  cudaError_t je = cudaEventRecord(hs->done, hs->d2h);
  if (je == cudaSuccess) je = cudaStreamWaitEvent(stream, hs->done, 0);
  if (st != SSM_OK) return st;
  return (e == cudaSuccess && je == cudaSuccess) ? SSM_OK : SSM_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* ssm_version(void) { return "0.1.0"; }

ssm_status ssm_selftest_wait_timeout(uint32_t polls, cudaStream_t stream) {
  if (polls > kSelftestMaxPolls) return SSM_ERR_SHAPE;
  int dev = 0;
  const ssm_status st = current_device_for(stream, &dev);
  if (st != SSM_OK) return st;
  return ssm::launch_wait_timeout_selftest(polls, stream) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

ssm_status ssm_check_device_errors(void) {
  unsigned int word = 0;
  if (!ssm::read_and_clear_device_errors(&word)) return SSM_ERR_CUDA;
  return word ? SSM_ERR_TIMEOUT : SSM_OK;
}

const char* ssm_status_string(ssm_status status) {
  switch (status) {
    case SSM_OK: return "ok";
    case SSM_ERR_NULL: return "a required pointer is NULL";
    case SSM_ERR_SHAPE: return "invalid or overflowing shape";
    case SSM_ERR_UNSUPPORTED: return "unsupported dstate, dtype, kernel tier or option";
    case SSM_ERR_ALIGN: return "pointer not aligned to its element size";
    case SSM_ERR_CUDA: return "CUDA launch or runtime error";
    case SSM_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

const char* ssm_kernel_name(ssm_kernel kernel) {
  switch (kernel) {
    case SSM_KERNEL_AUTO: return "auto";
    case SSM_KERNEL_SERIAL: return "serial";
    case SSM_KERNEL_WARPSCAN: return "warpscan";
    case SSM_KERNEL_STREAM: return "stream";
    case SSM_KERNEL_STREAM_TM: return "stream-tm";
  }
  return "unknown";
}

ssm_status ssm_ssd_fwd(const void* x, const void* delta, const float* A, const void* B,
                       const void* C, const float* D, const void* z, const int32_t* valid_len,
                       const float* h0, void* out_y, float* out_final_state,
                       const ssm_ssd_shapes* shapes, ssm_dtype dtype, cudaStream_t stream) {
  if (!shapes) return SSM_ERR_NULL;
  if (dtype != SSM_F32 && dtype != SSM_BF16) return SSM_ERR_UNSUPPORTED;
  const ssm_ssd_shapes& s = *shapes;
  if (s.batch < 1 || s.seqlen < 1 || s.nheads < 1 || s.headdim < 1 || s.dstate < 1)
    return SSM_ERR_SHAPE;
  if (dtype != SSM_BF16 || s.headdim != ssm::kSsdHeadDim || !ssm::ssd_supported_state(s.dstate))
    return SSM_ERR_UNSUPPORTED;
  int64_t dim, bl, bld, bln, bdn, bh;
  const int64_t lim = int64_t(1) << 60;
  if (!mul_ok(s.nheads, s.headdim, &dim) || !mul_ok(s.batch, s.seqlen, &bl) ||
      !mul_ok(bl, dim, &bld) || !mul_ok(bl, s.dstate, &bln) || !mul_ok(s.batch, dim, &bdn) ||
      !mul_ok(bdn, s.dstate, &bdn) || !mul_ok(s.batch, s.nheads, &bh) || bld > lim ||
      bln > lim || bdn > lim || bh > 0x7FFFFFFF)
    return SSM_ERR_SHAPE;
  if (!x || !delta || !A || !B || !C || !out_y) return SSM_ERR_NULL;
  if (!aligned(x, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(out_y, 16) ||
      (z && !aligned(z, 16)) || !aligned(delta, 2) || !aligned(A, 4) || (D && !aligned(D, 4)) ||
      (h0 && !aligned(h0, 4)) || (out_final_state && !aligned(out_final_state, 4)) ||
      (valid_len && !aligned(valid_len, 4)))
    return SSM_ERR_ALIGN;
  ssm::SsdParams p;
  p.x = x; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z;
  p.valid_len = valid_len; p.h0 = h0; p.y = out_y; p.h_final = out_final_state;
  p.batch = s.batch; p.seqlen = s.seqlen; p.nheads = s.nheads; p.headdim = s.headdim;
  p.dstate = s.dstate;
  int dev = 0;
  const ssm_status ds = current_device_for(stream, &dev);
  if (ds != SSM_OK) return ds;
  p.err = ssm::stream::error_word();
  if (!p.err) return SSM_ERR_CUDA;
  return ssm::launch_ssd(p, stream) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

int64_t ssm_chunk_count(const ssm_shapes* shapes) {
  if (shapes == nullptr || shapes->chunk_len <= 0 || shapes->seqlen < 1) return 0;
  return (shapes->seqlen + shapes->chunk_len - 1) / shapes->chunk_len;
}

ssm_status ssm_scan_plan(const ssm_shapes* shapes, ssm_dtype dtype, int has_z, int has_valid_len,
                         int has_states, const ssm_options* opts, ssm_kernel* kernel,
                         int64_t* grid_blocks) {
  ssm_status st = check_shapes(shapes, dtype, has_states != 0);
  if (st != SSM_OK) return st;
  if ((st = check_options(opts)) != SSM_OK) return st;
  // Placeholder pointers: planning looks only at shapes and which tensors exist.
  alignas(256) static const char dummy[256] = {0};
  ScanParams p = make_params(dummy, dummy, reinterpret_cast<const float*>(dummy), dummy, dummy,
                             nullptr, has_z ? dummy : nullptr,
                             has_valid_len ? reinterpret_cast<const int32_t*>(dummy) : nullptr,
                             const_cast<char*>(dummy),
                             has_states ? reinterpret_cast<float*>(const_cast<char*>(dummy)) : nullptr,
                             shapes);
  Plan plan;
  if ((st = make_plan(p, dtype, opts, &plan)) != SSM_OK) return st;
  if (kernel) *kernel = plan.kernel;
  if (grid_blocks) *grid_blocks = plan.grid;
  return SSM_OK;
}

ssm_status ssm_scan_fwd_ex(const void* x, const void* delta, const float* A, const void* B,
                           const void* C, const float* D, const void* z,
                           const int32_t* valid_len, void* out_y, float* out_chunk_states,
                           const ssm_shapes* shapes, ssm_dtype dtype, cudaStream_t stream,
                           const ssm_options* opts) {
  return ssm_scan_fwd_carry(x, delta, A, B, C, D, z, valid_len, nullptr, out_y, out_chunk_states,
                            nullptr, shapes, dtype, stream, opts);
}

ssm_status ssm_scan_fwd_carry(const void* x, const void* delta, const float* A, const void* B,
                              const void* C, const float* D, const void* z,
                              const int32_t* valid_len, const float* h0, void* out_y,
                              float* out_chunk_states, float* out_final_state,
                              const ssm_shapes* shapes, ssm_dtype dtype, cudaStream_t stream,
                              const ssm_options* opts) {
  return ssm_scan_fwd_prep(x, delta, nullptr, A, B, C, D, z, valid_len, h0, out_y,
                           out_chunk_states, out_final_state, shapes, dtype, stream, opts);
}

ssm_status ssm_scan_fwd_prep(const void* x, const void* delta, const ssm_delta_prep* prep,
                             const float* A, const void* B, const void* C, const float* D,
                             const void* z, const int32_t* valid_len, const float* h0,
                             void* out_y, float* out_chunk_states, float* out_final_state,
                             const ssm_shapes* shapes, ssm_dtype dtype, cudaStream_t stream,
                             const ssm_options* opts) {
  ssm_status st = check_shapes(shapes, dtype, out_chunk_states != nullptr);
  if (st != SSM_OK) return st;
  if ((st = check_options(opts)) != SSM_OK) return st;
  if (!x || !delta || !A || !B || !C || !out_y) return SSM_ERR_NULL;
  const size_t es = elem_size(dtype);
  if (!aligned(x, es) || !aligned(delta, es) || !aligned(B, es) || !aligned(C, es) ||
      !aligned(out_y, es) || (z && !aligned(z, es)) || !aligned(A, 4) || (D && !aligned(D, 4)) ||
      (valid_len && !aligned(valid_len, 4)) || (out_chunk_states && !aligned(out_chunk_states, 4)) ||
      (h0 && !aligned(h0, 4)) || (out_final_state && !aligned(out_final_state, 4)))
    return SSM_ERR_ALIGN;

  ScanParams p = make_params(x, delta, A, B, C, D, z, valid_len, out_y, out_chunk_states, shapes,
                             h0, out_final_state);
  if ((st = apply_prep(prep, &p)) != SSM_OK) return st;
  return launch(p, dtype, opts, stream);
}

}  // extern "C"

// ---- the time split of the forward ---------------------------------------------
namespace {

struct SplitPlan {
  int64_t segments, seg_len;
  size_t bytes, off_hend, off_dtsum, off_h0;
  ssm::StreamShape shape;
};

// Segments (0 = the library's choice), their length (whole 64-step tiles) and
// the workspace layout: per (batch row, segment) the end state from a zero
// start, the sum of delta, and the state carried into the segment.
ssm_status split_plan(const ScanParams& p, ssm_dtype dtype, int64_t requested, SplitPlan* out) {
  const bool bf16 = dtype == SSM_BF16;
  if (requested < 0) return SSM_ERR_SHAPE;
  const ssm::StreamShape sh1 = ssm::stream_shape(p, bf16, 0, 0, 0);
  if (!ssm::stream_eligible(p, bf16, sh1)) return SSM_ERR_UNSUPPORTED;
  int64_t segs = requested == 0 ? ssm::stream_auto_segments(p, sh1) : requested;
  const int64_t tiles = (p.seqlen + 63) / 64;
  if (segs > tiles) segs = tiles;
  const int64_t seg_len = ((p.seqlen + segs - 1) / segs + 63) / 64 * 64;
  segs = (p.seqlen + seg_len - 1) / seg_len;
  ScanParams q = p;  // the launch shape for batch * segments rows
  q.batch = p.batch * segs;
  const ssm::StreamShape sh = segs == 1 ? sh1 : ssm::stream_shape(q, bf16, 0, 0, 0);
  if (sh.g == 0 || ssm::stream_grid(q, sh) > INT32_MAX) return SSM_ERR_UNSUPPORTED;
  out->segments = segs;
  out->seg_len = segs == 1 ? 0 : seg_len;
  out->shape = sh;
  out->bytes = out->off_hend = out->off_dtsum = out->off_h0 = 0;
  if (segs > 1) {
    const size_t rows = size_t(p.batch) * segs;
    const size_t st = rows * size_t(p.dim) * p.dstate * 4;
    out->off_hend = 0;
    out->off_dtsum = round_up(st, 256);
    out->off_h0 = out->off_dtsum + round_up(rows * size_t(p.dim) * 4, 256);
    out->bytes = out->off_h0 + st;
  }
  return SSM_OK;
}

}  // namespace

extern "C" {

ssm_status ssm_scan_split_plan(const ssm_shapes* shapes, ssm_dtype dtype, int has_z,
                               int64_t time_segments, int64_t* segments,
                               size_t* workspace_bytes) {
  ssm_status st = check_shapes(shapes, dtype, false);
  if (st != SSM_OK) return st;
  alignas(256) static const char dummy[256] = {0};
  ScanParams p = make_params(dummy, dummy, reinterpret_cast<const float*>(dummy), dummy, dummy,
                             nullptr, has_z ? dummy : nullptr, nullptr, const_cast<char*>(dummy),
                             nullptr, shapes);
  SplitPlan plan;
  if ((st = split_plan(p, dtype, time_segments, &plan)) != SSM_OK) return st;
  if (segments) *segments = plan.segments;
  if (workspace_bytes) *workspace_bytes = plan.bytes;
  return SSM_OK;
}

ssm_status ssm_scan_fwd_split(const void* x, const void* delta, const float* A, const void* B,
                              const void* C, const float* D, const void* z,
                              const int32_t* valid_len, const float* h0, void* out_y,
                              float* out_chunk_states, float* out_final_state,
                              const ssm_shapes* shapes, ssm_dtype dtype, int64_t time_segments,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  ssm_status st = check_shapes(shapes, dtype, out_chunk_states != nullptr);
  if (st != SSM_OK) return st;
  if (!x || !delta || !A || !B || !C || !out_y) return SSM_ERR_NULL;
  const size_t es = elem_size(dtype);
  if (!aligned(x, es) || !aligned(delta, es) || !aligned(B, es) || !aligned(C, es) ||
      !aligned(out_y, es) || (z && !aligned(z, es)) || !aligned(A, 4) || (D && !aligned(D, 4)) ||
      (valid_len && !aligned(valid_len, 4)) || (out_chunk_states && !aligned(out_chunk_states, 4)) ||
      (h0 && !aligned(h0, 4)) || (out_final_state && !aligned(out_final_state, 4)))
    return SSM_ERR_ALIGN;
  ScanParams p = make_params(x, delta, A, B, C, D, z, valid_len, out_y, out_chunk_states, shapes,
                             h0, out_final_state);
  SplitPlan plan;
  if ((st = split_plan(p, dtype, time_segments, &plan)) != SSM_OK) return st;
  int dev = 0;
  if ((st = current_device_for(stream, &dev)) != SSM_OK) return st;
  const bool bf16 = dtype == SSM_BF16;
  if (plan.segments == 1)  // no split: the STREAM tier as it is
    return ssm::launch_stream(p, bf16, stream, plan.shape) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
  if (workspace == nullptr) return SSM_ERR_NULL;
  if (!aligned(workspace, 256)) return SSM_ERR_ALIGN;
  if (workspace_bytes < plan.bytes) return SSM_ERR_SHAPE;
  char* ws = static_cast<char*>(workspace);
  p.seg_len = plan.seg_len;
  p.n_seg = static_cast<int>(plan.segments);
  p.seg_hend = reinterpret_cast<float*>(ws + plan.off_hend);
  p.seg_dtsum = reinterpret_cast<float*>(ws + plan.off_dtsum);
  p.seg_h0 = reinterpret_cast<float*>(ws + plan.off_h0);
  cudaError_t e = ssm::launch_stream_agg(p, bf16, stream, plan.shape);  // aggregates
  if (e == cudaSuccess) e = ssm::launch_seg_carry(p, stream);           // carries
  if (e == cudaSuccess) e = ssm::launch_stream(p, bf16, stream, plan.shape);  // the outputs
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

ssm_status ssm_scan_fwd(const void* x, const void* delta, const float* A, const void* B,
                        const void* C, const float* D, const void* z, const int32_t* valid_len,
                        void* out_y, float* out_chunk_states, const ssm_shapes* shapes,
                        ssm_dtype dtype, cudaStream_t stream) {
  return ssm_scan_fwd_ex(x, delta, A, B, C, D, z, valid_len, out_y, out_chunk_states, shapes,
                         dtype, stream, nullptr);
}

size_t ssm_scan_host_workspace_bytes(const ssm_shapes* shapes, ssm_dtype dtype, int has_D,
                                     int has_z, int has_valid_len, int has_states) {
  if (check_shapes(shapes, dtype, has_states != 0) != SSM_OK) return 0;
  const size_t total = host_layout(shapes, dtype, has_D, has_z, has_valid_len, has_states).total;
  return total == kNoFit ? 0 : total;
}

ssm_status ssm_scan_fwd_host(const void* x, const void* delta, const float* A, const void* B,
                             const void* C, const float* D, const void* z,
                             const int32_t* valid_len, void* out_y, float* out_chunk_states,
                             const ssm_shapes* shapes, ssm_dtype dtype, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
  const bool want_states = out_chunk_states != nullptr;
  ssm_status st = check_shapes(shapes, dtype, want_states);
  if (st != SSM_OK) return st;
  if (!x || !delta || !A || !B || !C || !out_y || !workspace) return SSM_ERR_NULL;
  if (!aligned(workspace, 256)) return SSM_ERR_ALIGN;
  const HostLayout l = host_layout(shapes, dtype, D != nullptr, z != nullptr,
                                   valid_len != nullptr, want_states);
  if (l.total == kNoFit || workspace_bytes < l.total) return SSM_ERR_SHAPE;
  return run_host_pipeline(x, delta, A, B, C, D, z, valid_len, out_y, out_chunk_states, *shapes,
                           dtype, static_cast<char*>(workspace), l, stream);
}

ssm_status ssm_decode_step(const void* x, const void* delta, const float* A, const void* B,
                           const void* C, const float* D, const void* z, float* state,
                           void* out_y, int64_t batch, int64_t dim, int64_t dstate,
                           ssm_dtype dtype, cudaStream_t stream) {
  return ssm_decode_step_prep(x, delta, nullptr, A, B, C, D, z, state, out_y, batch, dim, dstate,
                              dtype, stream);
}

ssm_status ssm_decode_step_prep(const void* x, const void* delta, const ssm_delta_prep* prep,
                                const float* A, const void* B, const void* C, const float* D,
                                const void* z, float* state, void* out_y, int64_t batch,
                                int64_t dim, int64_t dstate, ssm_dtype dtype,
                                cudaStream_t stream) {
  if (dtype != SSM_F32 && dtype != SSM_BF16) return SSM_ERR_UNSUPPORTED;
  if (batch < 1 || dim < 1 || dstate < 1) return SSM_ERR_SHAPE;
  if (!supported_dstate(dstate)) return SSM_ERR_UNSUPPORTED;
  int64_t bd, bdn, dn;
  const int64_t lim = int64_t(1) << 60;
  if (!mul_ok(batch, dim, &bd) || !mul_ok(bd, dstate, &bdn) || !mul_ok(dim, dstate, &dn) ||
      bdn > lim || dn > lim || bd * 16 > lim)
    return SSM_ERR_SHAPE;
  if (!x || !delta || !A || !B || !C || !state || !out_y) return SSM_ERR_NULL;
  const size_t es = elem_size(dtype);
  if (!aligned(x, es) || !aligned(delta, es) || !aligned(B, es) || !aligned(C, es) ||
      !aligned(out_y, es) || (z && !aligned(z, es)) || (D && !aligned(D, 4)) ||
      !aligned(A, 16) || !aligned(state, 16))
    return SSM_ERR_ALIGN;
  ssm::DecodeParams p;
  p.x = x; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z;
  p.state = state; p.y = out_y;
  p.batch = batch; p.dim = dim; p.dstate = static_cast<int>(dstate);
  p.dt_bias = nullptr; p.delta_softplus = 0; p.delta_clamp = 0; p.delta_lo = 0.f; p.delta_hi = 0.f;
  const ssm_status st = apply_prep(prep, &p);
  if (st != SSM_OK) return st;
  return ssm::launch_decode(p, dtype == SSM_BF16, stream) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

ssm_status ssm_scan_bwd(const void* x, const void* delta, const float* A, const void* B,
                        const void* C, const float* D, const void* z,
                        const int32_t* valid_len, const float* h0, const float* chunk_states,
                        const void* dy, void* dx, void* ddelta, float* dA, float* dB, float* dC,
                        float* dD, void* dz, float* dh0, const ssm_shapes* shapes,
                        ssm_dtype dtype, cudaStream_t stream) {
  ssm_status st = check_shapes(shapes, dtype, true);
  if (st != SSM_OK) return st;
  if (shapes->chunk_len > kBwdMaxChunk) return SSM_ERR_UNSUPPORTED;
  if (!x || !delta || !A || !B || !C || !chunk_states || !dy || !dx || !ddelta || !dA || !dB ||
      !dC)
    return SSM_ERR_NULL;
  if (z && !dz) return SSM_ERR_NULL;
  const size_t es = elem_size(dtype);
  if (!aligned(x, es) || !aligned(delta, es) || !aligned(B, es) || !aligned(C, es) ||
      !aligned(dy, es) || !aligned(dx, es) || !aligned(ddelta, es) || (z && !aligned(z, es)) ||
      (dz && !aligned(dz, es)) || !aligned(A, 4) || (D && !aligned(D, 4)) ||
      (valid_len && !aligned(valid_len, 4)) || (h0 && !aligned(h0, 4)) ||
      !aligned(chunk_states, 4) || !aligned(dA, 4) || !aligned(dB, 4) || !aligned(dC, 4) ||
      (dD && !aligned(dD, 4)) || (dh0 && !aligned(dh0, 4)))
    return SSM_ERR_ALIGN;
  ssm::BwdParams p;
  p.fwd = make_params(x, delta, A, B, C, D, z, valid_len, nullptr,
                      const_cast<float*>(chunk_states), shapes, h0, nullptr);
  p.dy = dy; p.dx = dx; p.ddelta = ddelta; p.dz = z ? dz : nullptr;
  p.dA = dA; p.dB = dB; p.dC = dC; p.dD = D ? dD : nullptr; p.dh0 = dh0;
  const size_t bln = size_t(shapes->batch) * shapes->seqlen * shapes->dstate * sizeof(float);
  cudaError_t e = cudaMemsetAsync(dA, 0, size_t(shapes->dim) * shapes->dstate * sizeof(float),
                                  stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(dB, 0, bln, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(dC, 0, bln, stream);
  if (e == cudaSuccess && p.dD) e = cudaMemsetAsync(dD, 0, size_t(shapes->dim) * sizeof(float),
                                                    stream);
  if (e == cudaSuccess) e = ssm::launch_bwd(p, dtype == SSM_BF16, stream);
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

}  // extern "C"

// ---- the end-to-end form without any allocation ------------------------------------
//
// The same computation as ssm_scan_fwd_host (pieces chained by the carried
// state), with its device workspace in a fixed file-scope array instead of a
// caller-owned buffer, and every copy and kernel on the caller's stream (no
// library streams or events are created).

namespace {

constexpr size_t kStaticWsBytes = size_t(64) << 20;  // 64 MiB
__device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

// Address of g_static_ws on each device, looked up once with that device current.
char* static_ws(int dev) {
  static char* addr[64] = {};
  static std::mutex mu;
  if (dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (addr[dev] == nullptr) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_static_ws) != cudaSuccess || a == nullptr) return nullptr;
    addr[dev] = static_cast<char*>(a);
  }
  return addr[dev];
}

}  // namespace

extern "C" {

size_t ssm_scan_host_static_capacity(void) { return kStaticWsBytes; }

ssm_status ssm_scan_fwd_host_static(const void* x, const void* delta, const float* A,
                                    const void* B, const void* C, const float* D, const void* z,
                                    const int32_t* valid_len, void* out_y, float* out_chunk_states,
                                    const ssm_shapes* shapes, ssm_dtype dtype,
                                    cudaStream_t stream) {
  const bool want_states = out_chunk_states != nullptr;
  ssm_status st = check_shapes(shapes, dtype, want_states);
  if (st != SSM_OK) return st;
  if (!x || !delta || !A || !B || !C || !out_y) return SSM_ERR_NULL;
  const HostLayout l = host_layout(shapes, dtype, D != nullptr, z != nullptr,
                                   valid_len != nullptr, want_states);
  if (l.total == kNoFit || l.total > kStaticWsBytes)
    return SSM_ERR_SHAPE;  // larger than the fixed workspace
  int dev = 0;
  if ((st = current_device_for(stream, &dev)) != SSM_OK) return st;
  char* ws = static_ws(dev);
  if (ws == nullptr) return SSM_ERR_CUDA;

  const ssm_shapes& s = *shapes;
  const size_t es = elem_size(dtype);
  const int64_t L = s.seqlen, Bt = s.batch, N = s.dstate;
  const size_t dn4 = size_t(s.dim) * N * 4;
  const int64_t nch = want_states ? (L + s.chunk_len - 1) / s.chunk_len : 0;
  const int64_t piece = host_piece_steps(s, dtype, z != nullptr, want_states);
  float* carry[2] = {reinterpret_cast<float*>(ws + l.carry),
                     reinterpret_cast<float*>(ws + l.carry + size_t(Bt) * dn4)};
  cudaError_t e = cudaSuccess;
  auto ok = [&](cudaError_t r) { if (e == cudaSuccess) e = r; return e == cudaSuccess; };
  auto copy_in = [&](size_t region, const void* src, int64_t w, int64_t t0, int64_t n) {
    const size_t row = size_t(w) * es;
    return ok(cudaMemcpy2DAsync(ws + region + size_t(Bt) * t0 * row, n * row,
                                static_cast<const char*>(src) + t0 * row, L * row, n * row, Bt,
                                cudaMemcpyHostToDevice, stream));
  };
  // Nothing in the workspace has to start at zero: every piece's carried state
  // is written by the piece before it is read, and the first piece starts
  // from h0 = 0 without reading the workspace.
  ok(cudaMemcpyAsync(ws + l.A, A, dn4, cudaMemcpyHostToDevice, stream));
  if (D) ok(cudaMemcpyAsync(ws + l.D, D, size_t(s.dim) * 4, cudaMemcpyHostToDevice, stream));
  if (valid_len)
    ok(cudaMemcpyAsync(ws + l.valid, valid_len, size_t(Bt) * 4, cudaMemcpyHostToDevice, stream));
  int i = 0;
  for (int64_t t0 = 0; t0 < L && e == cudaSuccess; t0 += piece, ++i) {
    const int64_t n = L - t0 < piece ? L - t0 : piece;
    const size_t act_off = size_t(Bt) * t0 * s.dim * es, bc_off = size_t(Bt) * t0 * N * es;
    copy_in(l.x, x, s.dim, t0, n);
    copy_in(l.delta, delta, s.dim, t0, n);
    if (z) copy_in(l.z, z, s.dim, t0, n);
    copy_in(l.B, B, N, t0, n);
    copy_in(l.C, C, N, t0, n);
    if (e != cudaSuccess) break;
    const int64_t c0 = want_states ? t0 / s.chunk_len : 0;
    const int64_t pch = want_states ? (n + s.chunk_len - 1) / s.chunk_len : 0;
    float* pstates = want_states ? reinterpret_cast<float*>(ws + l.states) + size_t(Bt) * c0 *
                                       (dn4 / 4)
                                 : nullptr;
    const ssm_shapes ps = {Bt, n, s.dim, N, want_states ? s.chunk_len : 0};
    ScanParams p = make_params(ws + l.x + act_off, ws + l.delta + act_off,
                               reinterpret_cast<const float*>(ws + l.A), ws + l.B + bc_off,
                               ws + l.C + bc_off,
                               D ? reinterpret_cast<const float*>(ws + l.D) : nullptr,
                               z ? ws + l.z + act_off : nullptr,
                               valid_len ? reinterpret_cast<const int32_t*>(ws + l.valid) : nullptr,
                               ws + l.y + act_off, pstates, &ps,
                               t0 == 0 ? nullptr : carry[i % 2],
                               t0 + n < L ? carry[(i + 1) % 2] : nullptr);
    p.len_offset = t0;
    st = launch(p, dtype, nullptr, stream);
    if (st != SSM_OK) return st;
    const size_t row = size_t(s.dim) * es;
    ok(cudaMemcpy2DAsync(static_cast<char*>(out_y) + t0 * row, L * row, ws + l.y + act_off,
                         n * row, n * row, Bt, cudaMemcpyDeviceToHost, stream));
    if (want_states)
      ok(cudaMemcpy2DAsync(out_chunk_states + size_t(c0) * (dn4 / 4), nch * dn4, pstates,
                           pch * dn4, pch * dn4, Bt, cudaMemcpyDeviceToHost, stream));
  }
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

}  // extern "C"
