// tiers.h -- launchers of the kernel tiers, called by the C ABI layer (api.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace ssm {

// Correctness tier: one thread per (b, d); any supported shape.
cudaError_t launch_serial(const ScanParams& p, bool bf16, cudaStream_t s);
int64_t serial_grid(const ScanParams& p);

}  // namespace ssm
