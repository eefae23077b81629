/*
 * ssmscan.h -- C ABI of libssmscan, the fused selective-scan forward for
 * NVIDIA GB300 (sm_103a).
 *
 * What the library computes (page, then section):
 *   [P1] the article at pwwt.cn/news/6372990 on Mamba's hardware-aware
 *        algorithm and parallel associative scan;
 *   [P2] "Mamba并行扫描与硬件感知优化：从SSM递推到GPU高效实现"
 *        (bjdmk.com.cn/news/5218626).
 *
 * For every batch row b, channel d and state n, with h_{-1} = 0 ([P1] s4.1):
 *     a_t   = exp(delta[b,t,d] * A[d,n])              ([P1] s2.4: Abar = exp(delta A))
 *     h_t   = a_t * h_{t-1} + delta[b,t,d] * B[b,t,n] * x[b,t,d]
 *                                                     ([P1] s1.1 recurrence, s3.3 b = Bbar x)
 *     y[b,t,d] = (sum_n C[b,t,n] * h_t + D[d] * x[b,t,d]) * silu(z[b,t,d])
 *                                                     ([P1] s1.1 output and D residual;
 *                                                      the gate is optional)
 * The recurrence is evaluated as a parallel associative scan over (a, b)
 * pairs with the combine (a1,b1) o (a2,b2) = (a1 a2, a2 b1 + b2)
 * ([P1] s2.1, [P2] s2.2), or as a register-resident serial sweep where the
 * batch and channel dimensions already fill the GPU.  The state h stays in
 * registers: only x, delta, z, B, C, A, D are read and y (plus optional chunk
 * boundary states, [P1] s3.4) is written.
 *
 * Steps t >= valid_len[b] are the identity step (a = 1, b = 0, [P1] s2.3): the
 * state is frozen and y there is exactly 0.
 *
 * Conventions for every entry point below:
 *   - All tensors are dense, row-major, contiguous.  Shapes:
 *       x, delta, z, y : [batch, seqlen, dim]       dtype of the call
 *       B, C           : [batch, seqlen, dstate]    dtype of the call (shared by all d)
 *       A              : [dim, dstate]              fp32 (A < 0 expected, not required)
 *       D              : [dim]                      fp32
 *       valid_len      : [batch]                    int32
 *       chunk states   : [batch, ceil(seqlen/chunk_len), dim, dstate]  fp32
 *   - The caller owns every buffer; the library keeps no pointer after a call
 *     returns and allocates no device memory on this path.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream) and never
 *     synchronise the host.  Argument errors are detected on the host before
 *     any launch and are returned as a status; nothing is launched then.  A
 *     launch failure is returned as SSM_ERR_CUDA (cudaGetLastError() tells
 *     which).  No entry point aborts, throws or traps.
 *   - `stream` must belong to the calling thread's current device (checked,
 *     SSM_ERR_CUDA otherwise), except while it is being captured into a CUDA
 *     graph: the device entry points (forward, split, backward, decode, SSD)
 *     then only record their work, and the captured graph replays it.  Make one
 *     call of each shape outside the capture first (it performs the library's
 *     one-time lookups).
 *   - Inputs and outputs must not overlap.
 */
#ifndef SSMSCAN_H_
#define SSMSCAN_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SSM_OK = 0,
  SSM_ERR_NULL = 1,        /* a required pointer is NULL */
  SSM_ERR_SHAPE = 2,       /* a size is negative or zero where it must not be, or overflows */
  SSM_ERR_UNSUPPORTED = 3, /* dstate not in {1,2,4,8,16,32,64}, unknown dtype, kernel or flag */
  SSM_ERR_ALIGN = 4,       /* a pointer is not aligned to its element size */
  SSM_ERR_CUDA = 5,        /* a CUDA runtime call or a kernel launch failed */
  SSM_ERR_TIMEOUT = 6      /* reserved for bounded device-side waits */
} ssm_status;

/* Element type of x, delta, B, C, z and y.  A, D and the chunk states are
 * always fp32 and all arithmetic is fp32 ([P1] s2.4: the prefix is accumulated
 * in fp32 even when the inputs are bf16). */
typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype;

typedef struct {
  int64_t batch;     /* >= 1 */
  int64_t seqlen;    /* L >= 1 */
  int64_t dim;       /* channels D >= 1 */
  int64_t dstate;    /* N, one of 1, 2, 4, 8, 16, 32, 64 */
  int64_t chunk_len; /* steps per boundary-state chunk; 0 = no chunk states */
} ssm_shapes;

/* Kernel tiers.  AUTO picks the fastest eligible tier for the shape. */
typedef enum {
  SSM_KERNEL_AUTO = 0,
  SSM_KERNEL_SERIAL = 1,   /* one thread per (b, d), all N states serial; any shape */
  SSM_KERNEL_WARPSCAN = 2, /* [P1] s3.1 hierarchy: thread-serial run of k steps,
                              5-round shuffle scan across the warp, serial carry
                              between windows; one warp per (b, d) */
  SSM_KERNEL_STREAM = 3,   /* register sweep over channels x states per thread, TMA-staged
                              tiles, f32x2 math over channel pairs; needs
                              batch*dim*dstate to fill the GPU */
  SSM_KERNEL_STREAM_TM = 4 /* the register sweep with the B and C rows broadcast to every
                              thread through tensor memory by one exact tensor-core
                              product per group of steps ([P1] s3.2: B and C are shared by
                              all channels); one channel x 4 (dstate 16) or 8 (dstate 64)
                              states per thread, f32x2 math over state pairs; dstate 16
                              or 64, no fused step-size preparation, bf16 only with
                              dstate 16; no launch-shape options */
} ssm_kernel;

typedef struct {
  ssm_kernel kernel;       /* SSM_KERNEL_AUTO unless forcing a tier (tests, benchmarks) */
  int32_t warps_per_block;   /* 0 = the tier's default; STREAM accepts 1, 2 or 4 */
  int32_t states_per_lane;   /* 0 = the tier's default; STREAM: 4, 8 or 16 consecutive
                                states of a channel per thread (instances exist for some
                                (dstate, states, channels) combinations only) */
  int32_t channels_per_lane; /* 0 = the tier's default; STREAM: 2 or 4 consecutive
                                channels per thread, paired in f32x2 instructions */
} ssm_options;

/*
 * ssm_scan_fwd -- the fused selective-scan forward on device buffers.
 *
 *   x, delta, B, C : device, dtype `dtype`, required.
 *   A              : device fp32 [dim, dstate], required.
 *   D              : device fp32 [dim], or NULL for no D residual.
 *   z              : device, dtype `dtype`, or NULL for no gate.
 *   valid_len      : device int32 [batch], or NULL (every step valid).  Values
 *                    outside [0, seqlen] are clamped on the device.
 *   out_y          : device, dtype `dtype`, required.  bf16 results are rounded
 *                    to nearest even.
 *   out_chunk_states: device fp32, or NULL.  Written only when
 *                    shapes->chunk_len > 0: chunk c holds h at step
 *                    min((c+1)*chunk_len, seqlen) - 1 ([P1] s3.4).
 *   shapes         : host pointer, required.
 *   stream         : CUDA stream of the call.
 * Returns SSM_OK once the work is enqueued.
 */
ssm_status ssm_scan_fwd(const void* x, const void* delta, const float* A, const void* B,
                        const void* C, const float* D, const void* z, const int32_t* valid_len,
                        void* out_y, float* out_chunk_states, const ssm_shapes* shapes,
                        ssm_dtype dtype, cudaStream_t stream);

/* As ssm_scan_fwd, with an explicit kernel tier (opts may be NULL = AUTO).
 * A forced tier that cannot run the shape returns SSM_ERR_UNSUPPORTED. */
ssm_status ssm_scan_fwd_ex(const void* x, const void* delta, const float* A, const void* B,
                           const void* C, const float* D, const void* z,
                           const int32_t* valid_len, void* out_y, float* out_chunk_states,
                           const ssm_shapes* shapes, ssm_dtype dtype, cudaStream_t stream,
                           const ssm_options* opts);

/* The fused step-size preparation ([P1] s3.3: the fused kernel applies a bias,
 * softplus and lower/upper clipping to delta before the discretisation).  For
 * every (b, t, d), before delta is used:
 *   v = delta[b,t,d] + (dt_bias ? dt_bias[d] : 0)
 *   v = softplus ? ln(1 + e^v) : v
 *   v = clamp ? min(max(v, lo), hi) : v
 * Steps past valid_len stay the identity whatever the preparation gives.
 * dt_bias: device fp32 [dim] or NULL.  softplus, clamp: 0 or 1; with clamp,
 * lo <= hi is required. */
typedef struct {
  const float* dt_bias;
  int32_t softplus;
  int32_t clamp;
  float lo, hi;
} ssm_delta_prep;

/* As ssm_scan_fwd_ex, continuing from a given state and returning the final one.
 *   h0              : device fp32 [batch, dim, dstate], the state before the first
 *                     step (NULL = zeros, [P1] s4.1).
 *   out_final_state : device fp32 [batch, dim, dstate], receives the state after
 *                     the last step (frozen past valid_len), or NULL.
 * Running steps [0, k) and then [k, L) from the first call's final state gives
 * the same y and states as one call over [0, L): the serial carry between
 * chunks of the sequence ([P1] s3.1 third level, [P2] s2.4). */
ssm_status ssm_scan_fwd_carry(const void* x, const void* delta, const float* A, const void* B,
                              const void* C, const float* D, const void* z,
                              const int32_t* valid_len, const float* h0, void* out_y,
                              float* out_chunk_states, float* out_final_state,
                              const ssm_shapes* shapes, ssm_dtype dtype, cudaStream_t stream,
                              const ssm_options* opts);

/* The most general forward: ssm_scan_fwd_carry with the fused step-size
 * preparation `prep` (NULL = delta used as given).  Under SSM_KERNEL_AUTO the
 * STREAM tier runs it in its default launch shapes; forcing another STREAM
 * shape with a preparation returns SSM_ERR_UNSUPPORTED. */
ssm_status ssm_scan_fwd_prep(const void* x, const void* delta, const ssm_delta_prep* prep,
                             const float* A, const void* B, const void* C, const float* D,
                             const void* z, const int32_t* valid_len, const float* h0,
                             void* out_y, float* out_chunk_states, float* out_final_state,
                             const ssm_shapes* shapes, ssm_dtype dtype, cudaStream_t stream,
                             const ssm_options* opts);

/*
 * ssm_decode_step -- advance the recurrence by one step on a carried state
 * (token-by-token generation).  For every (b, d, n):
 *   h[b,d,n] <- exp(delta[b,d] A[d,n]) h[b,d,n] + delta[b,d] B[b,n] x[b,d]
 *   y[b,d]    = (sum_n C[b,n] h[b,d,n] + D[d] x[b,d]) * silu(z[b,d])
 * ([P1] s1.1, s2.4, s3.3): the scan of one step starting from `state`, with
 * the same fp32 arithmetic as ssm_scan_fwd, so that decoding a sequence step
 * by step follows its scan (SSM chunk carry [P1] s3.1, [P2] s2.4).
 *   x, delta, z : device, dtype `dtype`, [batch, dim] (z nullable: no gate).
 *   B, C        : device, dtype `dtype`, [batch, dstate].
 *   A           : device fp32 [dim, dstate], 16-byte aligned.  D: fp32 [dim] or NULL.
 *   state       : device fp32 [batch, dim, dstate], 16-byte aligned; read and
 *                 overwritten in place (typically the final state of a scan,
 *                 ssm_scan_fwd_carry).
 *   out_y       : device, dtype `dtype`, [batch, dim].
 * Asynchronous on `stream`; argument errors return a status before launch.
 */
ssm_status ssm_decode_step(const void* x, const void* delta, const float* A, const void* B,
                           const void* C, const float* D, const void* z, float* state,
                           void* out_y, int64_t batch, int64_t dim, int64_t dstate,
                           ssm_dtype dtype, cudaStream_t stream);

/* ssm_decode_step with the fused step-size preparation `prep` (NULL = none). */
ssm_status ssm_decode_step_prep(const void* x, const void* delta, const ssm_delta_prep* prep,
                                const float* A, const void* B, const void* C, const float* D,
                                const void* z, float* state, void* out_y, int64_t batch,
                                int64_t dim, int64_t dstate, ssm_dtype dtype,
                                cudaStream_t stream);

/*
 * ssm_scan_bwd -- the backward: every gradient of l = sum(dy * y) for the
 * forward ssm_scan_fwd_carry computes (delta used as given).
 *   Forward inputs x, delta, A, B, C, D, z, valid_len, h0: as in the forward.
 *   chunk_states : device fp32 [batch, ceil(L/chunk_len), dim, dstate], the
 *                  boundary states the forward wrote with the same chunk_len
 *                  (shapes->chunk_len, 1 .. 512); the backward replays the
 *                  forward from them ([P1] s3.4).
 *   dy           : device, dtype `dtype`, [batch, L, dim].
 *   dx, ddelta   : device, dtype `dtype`, [batch, L, dim] (outputs).
 *   dz           : device, dtype `dtype`, [batch, L, dim]; required with z.
 *   dA           : device fp32 [dim, dstate]; dB, dC: fp32 [batch, L, dstate];
 *                  dD: fp32 [dim] or NULL; all four are sums over channels,
 *                  steps or batch rows, zeroed on `stream` by the call.
 *   dh0          : device fp32 [batch, dim, dstate] or NULL: the gradient of
 *                  the state before the first step.
 * Steps past valid_len get zero gradients.  The summed outputs are added with
 * atomics: their last bits depend on the order.  Asynchronous on `stream`.
 * Kernel: with dstate 16, 32 or 64, chunk_len a multiple of 16, dim times the
 * element size a multiple of 16 bytes and every tensor 16-byte aligned, a
 * TMA-tiled kernel (the decays of each 16-step piece kept in registers, dB and
 * dC reduced in shared memory before the atomics); otherwise a generic kernel
 * with the same results within the same tolerance.
 */
ssm_status ssm_scan_bwd(const void* x, const void* delta, const float* A, const void* B,
                        const void* C, const float* D, const void* z,
                        const int32_t* valid_len, const float* h0, const float* chunk_states,
                        const void* dy, void* dx, void* ddelta, float* dA, float* dB, float* dC,
                        float* dD, void* dz, float* dh0, const ssm_shapes* shapes,
                        ssm_dtype dtype, cudaStream_t stream);

/*
 * ssm_ssd_fwd -- the state-space-duality (SSD) form of the scan, computed
 * blockwise with tensor-core matrix products ([P2] s5.1-s5.2: the recurrence
 * expanded into a semiseparable matrix product; blocks of steps by matrix
 * products, the state carried from block to block by the recurrence).  The
 * decay is shared by all channels and states of a head: the channels
 * d = h * headdim + p of head h use one step size delta[b,t,h] and one scalar
 * A[h] < 0.  For every (b, d, n), from h = h0 (zeros when NULL):
 *   h[b,d,n] <- exp(delta[b,t,h] A[h]) h[b,d,n] + delta[b,t,h] B[b,t,n] x[b,t,d]
 *   y[b,t,d]  = (sum_n C[b,t,n] h[b,d,n] + D[d] x[b,t,d]) * silu(z[b,t,d])
 * Steps t >= valid_len[b] are the identity and their output is exactly 0.
 *   x, z      : device bf16 [batch, seqlen, nheads*headdim], 16-byte aligned
 *               (z NULL: no gate).
 *   delta     : device bf16 [batch, seqlen, nheads], the step size as given (> 0).
 *   A         : device fp32 [nheads].  D: device fp32 [nheads*headdim] or NULL.
 *   B, C      : device bf16 [batch, seqlen, dstate], 16-byte aligned.
 *   valid_len : device int32 [batch] or NULL; clamped to [0, seqlen] on the device.
 *   h0        : device fp32 [batch, nheads*headdim, dstate] or NULL.
 *   out_y     : device bf16 [batch, seqlen, nheads*headdim], 16-byte aligned.
 *   out_final_state : device fp32 [batch, nheads*headdim, dstate], the state
 *               after the last step, or NULL.
 * Supported: dtype SSM_BF16, headdim 64, dstate 128 or 256; other sizes or fp32
 * return SSM_ERR_UNSUPPORTED.  The products take bf16 operands (the inputs, the masked
 * decay-weighted block matrix and the state entering a block, rounded to bf16)
 * and accumulate in fp32; the state between blocks of 128 steps stays fp32.
 * All pointers are caller-owned; nothing is allocated.  Asynchronous on
 * `stream`; argument errors return a status before launch (an empty sequence,
 * seqlen 0, is SSM_ERR_SHAPE, as for the scan).  A CTA whose
 * bounded wait on the tensor cores gives up sets the sticky device error word
 * (ssm_check_device_errors returns SSM_ERR_TIMEOUT; outputs undefined).
 */
typedef struct {
  int64_t batch, seqlen, nheads, headdim, dstate;
} ssm_ssd_shapes;

ssm_status ssm_ssd_fwd(const void* x, const void* delta, const float* A, const void* B,
                       const void* C, const float* D, const void* z, const int32_t* valid_len,
                       const float* h0, void* out_y, float* out_final_state,
                       const ssm_ssd_shapes* shapes, ssm_dtype dtype, cudaStream_t stream);

/*
 * ssm_scan_fwd_split -- the forward with its sequence split across CTAs
 * (the time split: [P1] s3.1's cross-block level, [P1] s4.2 the per-chunk
 * aggregates, their scan and the fix-up; [P2] s2.3-2.4).
 *
 * Each batch row is cut into `segments` segments of whole 64-step tiles.
 * Three launches on `stream`:
 *   1. the aggregate pass: every segment but the last runs the recurrence
 *      only (no C, no y) from a zero state (the first from h0) and leaves its
 *      end state and its sum of delta over the valid steps;
 *   2. the carry: per (b, d, n), the state entering segment s is
 *      h_s = exp(A sum(delta of s-1)) h_{s-1} + end_{s-1}, the composition of
 *      the segments' (prod a, b) aggregates under the scan's combine;
 *   3. the output pass: every segment runs the full forward from its carried
 *      state, so y, the chunk states and the final state are those of one
 *      unsplit run up to the rounding of the carried states (the decay of a
 *      segment is formed once from its sum of delta).
 * The aggregate pass costs about half an output pass over all but the last
 * segment; the split pays where batch * dim * dstate leaves most of the GPU
 * idle (long sequences of few channels).
 *
 *   h0, out_final_state: as ssm_scan_fwd_carry (nullable).
 *   time_segments: 0 = the library's choice (1 when the rows already fill the
 *                  GPU), else the requested count, rounded to whole tiles.
 *   workspace:     device memory of at least the bytes ssm_scan_split_plan
 *                  reports, 256-byte aligned, owned by the caller and unused
 *                  by other work until `stream` passes this call; NULL when
 *                  the plan has one segment.
 * The forward is the STREAM tier's (its dstate, alignment and size rules);
 * shapes it does not take return SSM_ERR_UNSUPPORTED.  Other arguments and
 * the outputs are those of ssm_scan_fwd_carry.
 */
ssm_status ssm_scan_fwd_split(const void* x, const void* delta, const float* A, const void* B,
                              const void* C, const float* D, const void* z,
                              const int32_t* valid_len, const float* h0, void* out_y,
                              float* out_chunk_states, float* out_final_state,
                              const ssm_shapes* shapes, ssm_dtype dtype, int64_t time_segments,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* The segment count ssm_scan_fwd_split would use for these shapes and
 * `time_segments` (0 = the library's choice, which depends on the current
 * device's SM count) and the workspace bytes it needs (0 for one segment).
 * Either output may be NULL. */
ssm_status ssm_scan_split_plan(const ssm_shapes* shapes, ssm_dtype dtype, int has_z,
                               int64_t time_segments, int64_t* segments,
                               size_t* workspace_bytes);

/* The tier (and its grid) that ssm_scan_fwd_ex would launch for these
 * arguments, without launching anything.  `has_*` describe which optional
 * tensors the call passes.  Writes the tier to *kernel and the launch grid
 * (number of thread blocks) to *grid_blocks; either output may be NULL. */
ssm_status ssm_scan_plan(const ssm_shapes* shapes, ssm_dtype dtype, int has_z, int has_valid_len,
                         int has_states, const ssm_options* opts, ssm_kernel* kernel,
                         int64_t* grid_blocks);

/*
 * ssm_scan_fwd_host -- the same forward on HOST buffers (end-to-end form).
 *
 * Every tensor pointer is a host pointer with the layout above (pinned memory
 * gives asynchronous copies; pageable memory works but copies synchronously).
 * The call copies the inputs into `workspace` (device memory owned by the
 * caller, at least ssm_scan_host_workspace_bytes() bytes, 256-byte aligned),
 * runs the forward there, and copies y (and the chunk states when requested)
 * back to out_y / out_chunk_states.  It returns once the work is enqueued;
 * the host buffers must stay valid, and the workspace unused by other work,
 * until `stream` reaches that point (synchronise `stream` before reading the
 * outputs).
 *
 * The work is pipelined over pieces of the sequence: the inputs of piece i+1
 * are copied in while piece i runs and piece i-1's outputs are copied out, on
 * two library-owned copy streams per device chained to `stream` by events;
 * each piece starts from the state the previous one ended in ([P1] s3.1 third
 * level, [P2] s2.4), so the result equals ssm_scan_fwd's on the same inputs.
 * Calls on the same device enqueue one at a time (a lock); the calling
 * thread's current device is used.
 */
ssm_status ssm_scan_fwd_host(const void* x, const void* delta, const float* A, const void* B,
                             const void* C, const float* D, const void* z,
                             const int32_t* valid_len, void* out_y, float* out_chunk_states,
                             const ssm_shapes* shapes, ssm_dtype dtype, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/*
 * ssm_scan_fwd_host_static -- ssm_scan_fwd_host without any allocation.  The
 * pages have no counterpart: this is a deployment form of the end-to-end call
 * for callers that may not allocate device memory (fixed-memory services).
 * The device workspace is a fixed array inside the library of
 * ssm_scan_host_static_capacity() bytes (64 MiB); calls whose workspace
 * (ssm_scan_host_workspace_bytes) is larger return SSM_ERR_SHAPE.  Every copy
 * and kernel runs on `stream` in order (no pipelining, no library streams or
 * events); the call allocates nothing, neither with cudaMalloc nor through
 * any other library.  Nothing in the array has to start at zero.
 *   - The array is shared by all calls on a device: calls that overlap in
 *     time (on different streams, or from several threads) race on it and
 *     must be serialised by the caller.
 *   - The first call on a device looks the array's address up (one runtime
 *     query); make it before capturing `stream` into a CUDA graph.
 * Arguments, layouts and the result are those of ssm_scan_fwd_host.
 */
ssm_status ssm_scan_fwd_host_static(const void* x, const void* delta, const float* A,
                                    const void* B, const void* C, const float* D, const void* z,
                                    const int32_t* valid_len, void* out_y, float* out_chunk_states,
                                    const ssm_shapes* shapes, ssm_dtype dtype,
                                    cudaStream_t stream);

/* Bytes of the fixed workspace of ssm_scan_fwd_host_static. */
size_t ssm_scan_host_static_capacity(void);

/* Device bytes ssm_scan_fwd_host needs for these shapes and optional tensors;
 * 0 on invalid shapes. */
size_t ssm_scan_host_workspace_bytes(const ssm_shapes* shapes, ssm_dtype dtype, int has_D,
                                     int has_z, int has_valid_len, int has_states);

/* Number of boundary-state chunks, ceil(seqlen / chunk_len); 0 when
 * chunk_len <= 0 or shapes is NULL. */
int64_t ssm_chunk_count(const ssm_shapes* shapes);

/* Static, human-readable text for a status / a kernel tier. */
const char* ssm_status_string(ssm_status status);
const char* ssm_kernel_name(ssm_kernel kernel);

/* Reads and clears the library's sticky device error word.  A kernel whose
 * bounded wait on a copy gives up sets it and returns early (its outputs are
 * then undefined).  Synchronises the current device.  Returns SSM_OK,
 * SSM_ERR_TIMEOUT, or SSM_ERR_CUDA if the word cannot be read. */
ssm_status ssm_check_device_errors(void);

/* Self-test of the error path of the bounded device waits (no page
 * counterpart: a diagnostic).  Launches, on `stream`, one thread that waits
 * with the kernels' bounded wait on an mbarrier nothing ever arrives on (no
 * copy or matrix product targets it, so nothing is in flight when it
 * returns); after `polls` unsuccessful polls it gives up and sets the sticky
 * error word.  A following ssm_check_device_errors() then returns
 * SSM_ERR_TIMEOUT (and clears the word); the GPU context stays usable.
 * polls > 2^20 returns SSM_ERR_SHAPE; a stream of another device than the
 * current one returns SSM_ERR_CUDA. */
ssm_status ssm_selftest_wait_timeout(uint32_t polls, cudaStream_t stream);

/* Library version, e.g. "0.1.0". */
const char* ssm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SSMSCAN_H_ */
