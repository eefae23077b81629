// stream_tmem_launch.cuh -- the launcher template of the STREAM-TM tier,
// included by the instance units stream_tmem_inst_n*.cu.
#pragma once

#include "stream_tmem.cuh"

namespace ssm {
namespace stream {
bool make_map(CUtensorMap* m, const void* base, bool bf16, int64_t inner, int64_t L, int64_t batch,
              int box_inner, int box_t);
unsigned int* error_word();
}  // namespace stream

namespace stream_tm {

// Dynamic shared memory of one CTA: the ring, the product operands, the
// partial-sum buffers, the barriers, and 1 KB of alignment slack.  At least
// 116 KB are requested so that one CTA holds an SM (its 512 TMEM columns are
// all there are).
template <class K>
int smem_bytes(int stages) {
  const int need = 1024 + stages * K::STAGE + K::KS * K::ABYTES + 2 * K::KS * K::OBYTES +
                   K::W * K::PBYTES + (2 * stages + 4) * 8 + 16;
  return need > 116 * 1024 ? need : 116 * 1024;
}

template <class K>
cudaError_t launch_k(const ScanParams& p, cudaStream_t s, int stages) {
  const bool bf16 = sizeof(typename K::IO) == 2;
  CUtensorMap mx, mdt, mz, mb, mc;
  if (!stream::make_map(&mx, p.x, bf16, p.dim, p.seqlen, p.batch, K::CW, K::T) ||
      !stream::make_map(&mdt, p.delta, bf16, p.dim, p.seqlen, p.batch, K::CW, K::T) ||
      !stream::make_map(&mb, p.B, bf16, K::N, p.seqlen, p.batch, K::N, K::T) ||
      !stream::make_map(&mc, p.C, bf16, K::N, p.seqlen, p.batch, K::N, K::T))
    return cudaErrorInvalidValue;
  if constexpr (K::GATE) {
    if (!stream::make_map(&mz, p.z, bf16, p.dim, p.seqlen, p.batch, K::CW, K::T))
      return cudaErrorInvalidValue;
  } else {
    mz = mx;  // unused
  }
  LaunchArgs la;
  la.stages = stages;
  la.err = stream::error_word();
  if (la.err == nullptr) return cudaErrorInvalidValue;
  const int smem = smem_bytes<K>(stages);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  static bool attr_done = false;
  if (!attr_done) {
    const cudaError_t e = cudaFuncSetAttribute(
        stream_tm_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int64_t cpc = int64_t(K::CW) * K::W;
  const int64_t grid = (p.dim + cpc - 1) / cpc * p.batch;
  stream_tm_kernel<K><<<static_cast<unsigned>(grid), (K::W + 1) * 32, smem, s>>>(mx, mdt, mz, mb, mc,
                                                                                 p, la);
  return cudaGetLastError();
}

template <int N, int G, int R, int W>
cudaError_t launch_impl(const ScanParams& p, bool bf16, cudaStream_t s, int stages) {
  if (bf16) {
    if constexpr ((32 / (N / G)) * R * 2 % 16 == 0)
      return p.z ? launch_k<Cfg<N, G, R, W, __nv_bfloat16, true>>(p, s, stages)
                 : launch_k<Cfg<N, G, R, W, __nv_bfloat16, false>>(p, s, stages);
    else
      return cudaErrorInvalidValue;
  }
  return p.z ? launch_k<Cfg<N, G, R, W, float, true>>(p, s, stages)
             : launch_k<Cfg<N, G, R, W, float, false>>(p, s, stages);
}

template <int N, int G, int R, int W>
int smem_impl(bool bf16, bool gate, int stages) {
  if (bf16) {
    if constexpr ((32 / (N / G)) * R * 2 % 16 == 0)
      return gate ? smem_bytes<Cfg<N, G, R, W, __nv_bfloat16, true>>(stages)
                  : smem_bytes<Cfg<N, G, R, W, __nv_bfloat16, false>>(stages);
    else
      return 0;
  }
  return gate ? smem_bytes<Cfg<N, G, R, W, float, true>>(stages)
              : smem_bytes<Cfg<N, G, R, W, float, false>>(stages);
}

template <int N, int G, int R, int W>
cudaError_t launch_ngw(const ScanParams& p, bool bf16, cudaStream_t s, int stages);
template <int N, int G, int R, int W>
int smem_ngw(bool bf16, bool gate, int stages);

#define SSM_TM_DEFINE(N_, G_, R_, W_)                                                                \
  template <>                                                                                        \
  cudaError_t launch_ngw<N_, G_, R_, W_>(const ScanParams& p, bool bf16, cudaStream_t s, int st) {  \
    return launch_impl<N_, G_, R_, W_>(p, bf16, s, st);                                              \
  }                                                                                                  \
  template <>                                                                                        \
  int smem_ngw<N_, G_, R_, W_>(bool bf16, bool gate, int st) {                                       \
    return smem_impl<N_, G_, R_, W_>(bf16, gate, st);                                                \
  }

}  // namespace stream_tm
}  // namespace ssm
