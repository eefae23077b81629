// api.cu -- the C ABI of libssmscan (declared in include/ssmscan.h).
//
// Host-side only: argument validation, choice of kernel tier, launch.  Every
// argument error is found here, before anything is enqueued, and is returned
// as an ssm_status; nothing aborts or throws across the ABI.
#include <cuda_runtime.h>
#include <stdint.h>

#include <new>

#include "ssmscan.h"
#include "tiers.h"

namespace {

using ssm::ScanParams;

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
  if (o->kernel < SSM_KERNEL_AUTO || o->kernel > SSM_KERNEL_STREAM) return SSM_ERR_UNSUPPORTED;
  if (o->states_per_lane != 0 && o->states_per_lane != 2 && o->states_per_lane != 4 &&
      o->states_per_lane != 8 && o->states_per_lane != 16)
    return SSM_ERR_UNSUPPORTED;
  if (o->time_split != 0 && o->time_split != 1 && o->time_split != 2) return SSM_ERR_UNSUPPORTED;
  return SSM_OK;
}

struct Plan {
  ssm_kernel kernel;
  int64_t grid;
  ssm::StreamShape shape;
};

// Tier choice.  `forced` is the caller's request (AUTO = let the library pick).
ssm_status make_plan(const ScanParams& p, ssm_dtype dtype, const ssm_options* o, Plan* out) {
  const bool bf16 = dtype == SSM_BF16;
  const ssm_kernel forced = o ? o->kernel : SSM_KERNEL_AUTO;
  const ssm::StreamShape shape =
      ssm::stream_shape(p, o ? o->warps_per_block : 0, o ? o->states_per_lane : 0,
                        o ? o->time_split : 0);
  ssm_kernel k = forced;
  if (k == SSM_KERNEL_AUTO)
    k = ssm::stream_eligible(p, bf16, shape) ? SSM_KERNEL_STREAM : SSM_KERNEL_SERIAL;
  out->kernel = k;
  out->shape = shape;
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
    default:
      return SSM_ERR_UNSUPPORTED;
  }
}

ScanParams make_params(const void* x, const void* delta, const float* A, const void* B,
                       const void* C, const float* D, const void* z, const int32_t* valid_len,
                       void* y, float* states, const ssm_shapes* s) {
  ScanParams p;
  p.x = x; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z;
  p.valid_len = valid_len; p.y = y;
  p.batch = s->batch; p.seqlen = s->seqlen; p.dim = s->dim;
  p.dstate = static_cast<int>(s->dstate);
  const bool st = states != nullptr && s->chunk_len > 0;
  p.states = st ? states : nullptr;
  p.chunk_len = st ? s->chunk_len : 1;
  p.n_chunks = st ? (s->seqlen + s->chunk_len - 1) / s->chunk_len : 0;
  return p;
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Byte layout of the device workspace used by ssm_scan_fwd_host.
struct HostLayout {
  size_t x, delta, z, B, C, A, D, valid, y, states, total;
};

HostLayout host_layout(const ssm_shapes* s, ssm_dtype dtype, int has_D, int has_z, int has_valid,
                       int has_states) {
  const size_t es = elem_size(dtype);
  const size_t act = size_t(s->batch) * s->seqlen * s->dim * es;
  const size_t bc = size_t(s->batch) * s->seqlen * s->dstate * es;
  const size_t nch = s->chunk_len > 0 ? size_t((s->seqlen + s->chunk_len - 1) / s->chunk_len) : 0;
  HostLayout l;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = round_up(off + bytes, 256); return o; };
  l.x = take(act);
  l.delta = take(act);
  l.z = has_z ? take(act) : 0;
  l.B = take(bc);
  l.C = take(bc);
  l.A = take(size_t(s->dim) * s->dstate * 4);
  l.D = has_D ? take(size_t(s->dim) * 4) : 0;
  l.valid = has_valid ? take(size_t(s->batch) * 4) : 0;
  l.y = take(act);
  l.states = has_states ? take(size_t(s->batch) * nch * s->dim * s->dstate * 4) : 0;
  l.total = off;
  return l;
}

}  // namespace

extern "C" {

const char* ssm_version(void) { return "0.1.0"; }

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
  }
  return "unknown";
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
  ssm_status st = check_shapes(shapes, dtype, out_chunk_states != nullptr);
  if (st != SSM_OK) return st;
  if ((st = check_options(opts)) != SSM_OK) return st;
  if (!x || !delta || !A || !B || !C || !out_y) return SSM_ERR_NULL;
  const size_t es = elem_size(dtype);
  if (!aligned(x, es) || !aligned(delta, es) || !aligned(B, es) || !aligned(C, es) ||
      !aligned(out_y, es) || (z && !aligned(z, es)) || !aligned(A, 4) || (D && !aligned(D, 4)) ||
      (valid_len && !aligned(valid_len, 4)) || (out_chunk_states && !aligned(out_chunk_states, 4)))
    return SSM_ERR_ALIGN;

  const ScanParams p = make_params(x, delta, A, B, C, D, z, valid_len, out_y, out_chunk_states,
                                   shapes);
  Plan plan;
  if ((st = make_plan(p, dtype, opts, &plan)) != SSM_OK) return st;
  const bool bf16 = dtype == SSM_BF16;
  cudaError_t err = cudaErrorInvalidValue;
  switch (plan.kernel) {
    case SSM_KERNEL_SERIAL: err = ssm::launch_serial(p, bf16, stream); break;
    case SSM_KERNEL_STREAM: err = ssm::launch_stream(p, bf16, stream, plan.shape); break;
    case SSM_KERNEL_WARPSCAN: err = ssm::launch_warpscan(p, bf16, stream); break;
    default: return SSM_ERR_UNSUPPORTED;
  }
  return err == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
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
  return host_layout(shapes, dtype, has_D, has_z, has_valid_len, has_states).total;
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
  if (workspace_bytes < l.total) return SSM_ERR_SHAPE;
  char* ws = static_cast<char*>(workspace);
  const size_t es = elem_size(dtype);
  const size_t act = size_t(shapes->batch) * shapes->seqlen * shapes->dim * es;
  const size_t bc = size_t(shapes->batch) * shapes->seqlen * shapes->dstate * es;
  const size_t nch = size_t(ssm_chunk_count(shapes));
  const size_t states_bytes = size_t(shapes->batch) * nch * shapes->dim * shapes->dstate * 4;

  auto h2d = [&](size_t off, const void* src, size_t bytes) {
    return cudaMemcpyAsync(ws + off, src, bytes, cudaMemcpyHostToDevice, stream);
  };
  cudaError_t e = cudaSuccess;
  if (e == cudaSuccess) e = h2d(l.x, x, act);
  if (e == cudaSuccess) e = h2d(l.delta, delta, act);
  if (e == cudaSuccess && z) e = h2d(l.z, z, act);
  if (e == cudaSuccess) e = h2d(l.B, B, bc);
  if (e == cudaSuccess) e = h2d(l.C, C, bc);
  if (e == cudaSuccess) e = h2d(l.A, A, size_t(shapes->dim) * shapes->dstate * 4);
  if (e == cudaSuccess && D) e = h2d(l.D, D, size_t(shapes->dim) * 4);
  if (e == cudaSuccess && valid_len) e = h2d(l.valid, valid_len, size_t(shapes->batch) * 4);
  if (e != cudaSuccess) return SSM_ERR_CUDA;

  st = ssm_scan_fwd(ws + l.x, ws + l.delta, reinterpret_cast<const float*>(ws + l.A), ws + l.B,
                    ws + l.C, D ? reinterpret_cast<const float*>(ws + l.D) : nullptr,
                    z ? ws + l.z : nullptr,
                    valid_len ? reinterpret_cast<const int32_t*>(ws + l.valid) : nullptr,
                    ws + l.y, want_states ? reinterpret_cast<float*>(ws + l.states) : nullptr,
                    shapes, dtype, stream);
  if (st != SSM_OK) return st;
  e = cudaMemcpyAsync(out_y, ws + l.y, act, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess && want_states && states_bytes > 0)
    e = cudaMemcpyAsync(out_chunk_states, ws + l.states, states_bytes, cudaMemcpyDeviceToHost,
                        stream);
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

}  // extern "C"
