// ssd.h -- device-side parameters and launcher of the SSD (one decay per
// head) form of the scan, computed blockwise with tensor-core matrix products.
#pragma once
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace ssm {

struct SsdParams {
  const void* x;      // [batch, seqlen, nheads * headdim], bf16
  const void* delta;  // [batch, seqlen, nheads], bf16, the step size as given
  const float* A;     // [nheads]
  const void* B;      // [batch, seqlen, dstate], bf16
  const void* C;      // [batch, seqlen, dstate], bf16
  const float* D;     // [nheads * headdim] or null
  const void* z;      // [batch, seqlen, nheads * headdim], bf16, or null (no gate)
  const int32_t* valid_len;  // [batch] or null
  const float* h0;    // [batch, nheads * headdim, dstate] or null
  void* y;            // [batch, seqlen, nheads * headdim], bf16
  float* h_final;     // [batch, nheads * headdim, dstate] or null
  int64_t batch, seqlen, nheads, headdim, dstate;
  unsigned int* err;  // sticky error word of the bounded waits
};

// Steps per block (the M of every product), and the supported head and state sizes.
constexpr int kSsdChunk = 128;
constexpr int kSsdHeadDim = 64;
inline bool ssd_supported_state(int64_t n) { return n == 128 || n == 256; }

size_t ssd_smem_bytes(int64_t dstate);

namespace stream {
unsigned int* error_word();  // the library's sticky device error word (kernel_stream.cu)
}
cudaError_t launch_ssd(const SsdParams& p, cudaStream_t s);

}  // namespace ssm
