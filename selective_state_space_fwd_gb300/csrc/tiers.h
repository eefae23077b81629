// tiers.h -- launchers of the kernel tiers, called by the C ABI layer (api.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace ssm {

// Correctness tier: one thread per (b, d); any supported shape.
cudaError_t launch_serial(const ScanParams& p, bool bf16, cudaStream_t s);
int64_t serial_grid(const ScanParams& p);

// STREAM tier: channel-pair register sweep with TMA-staged tiles.
struct StreamShape {
  int wpc;     // warps per thread block
  int g;       // states per lane
  int r;       // channels per lane
  int stages;  // slots in the shared-memory ring
};
// The launch shape for a request (0 = default); all zero when no instance exists.
StreamShape stream_shape(const ScanParams& p, bool bf16, int warps_per_block, int states_per_lane,
                         int channels_per_lane);
bool stream_eligible(const ScanParams& p, bool bf16, StreamShape sh);
int64_t stream_grid(const ScanParams& p, StreamShape sh);
cudaError_t launch_stream(const ScanParams& p, bool bf16, cudaStream_t s, StreamShape sh);
// Time split of STREAM: the aggregate pass (segments' end states from a zero
// start and their sums of delta) and the carry between segments.
cudaError_t launch_stream_agg(const ScanParams& p, bool bf16, cudaStream_t s, StreamShape sh);
cudaError_t launch_seg_carry(const ScanParams& p, cudaStream_t s);
// The number of segments the library picks for a row layout (1 = no split).
int64_t stream_auto_segments(const ScanParams& p, StreamShape sh);

// STREAM-TM tier: the register sweep with B and C broadcast through tensor memory.
struct StreamTmShape {
  int g;       // states per lane
  int r;       // channels per lane: 1 (f32x2 over state pairs) or 2 (over the channel pair)
  int warps;   // compute warps per thread block
  int stages;  // slots in the shared-memory ring
};
StreamTmShape stream_tm_shape(const ScanParams& p, bool bf16, int channels_per_lane);
bool stream_tm_eligible(const ScanParams& p, bool bf16, StreamTmShape sh);
int64_t stream_tm_grid(const ScanParams& p, StreamTmShape sh);
cudaError_t launch_stream_tm(const ScanParams& p, bool bf16, cudaStream_t s, StreamTmShape sh);

// WARPSCAN tier: one warp per (b, d), lanes along time, 5-round shuffle scan.
bool warpscan_eligible(const ScanParams& p);
int64_t warpscan_grid(const ScanParams& p);
cudaError_t launch_warpscan(const ScanParams& p, bool bf16, cudaStream_t s);

// Decode step: one step of the recurrence on a carried state, in place.
cudaError_t launch_decode(const DecodeParams& p, bool bf16, cudaStream_t s);

// Backward: every gradient of sum(dy * y), replaying the forward from its
// chunk boundary states.
cudaError_t launch_bwd(const BwdParams& p, bool bf16, cudaStream_t s);
size_t bwd_smem_bytes(int64_t chunk_len, int dstate);
// Its TMA-tiled form (16, 32 or 64 states, chunks a multiple of 16 steps,
// 16-byte aligned buffers); launch_bwd takes it whenever it is eligible.
bool bwd_tiled_eligible(const BwdParams& p, bool bf16);
cudaError_t launch_bwd_tiled(const BwdParams& p, bool bf16, cudaStream_t s);

// One thread runs a bounded wait on an mbarrier nothing arrives on, gives up
// after `polls` polls and sets the sticky error word (test of the error path).
cudaError_t launch_wait_timeout_selftest(unsigned polls, cudaStream_t s);

// Sticky device error word of the tiers with bounded waits: read and clear.
bool read_and_clear_device_errors(unsigned int* word);

}  // namespace ssm
