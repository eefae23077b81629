// STREAM instances for 64 states (kernel template in stream_core.cuh).
#include "stream_core.cuh"

namespace ssm {
namespace stream {
SSM_STREAM_DEFINE(64, 8, 2)
SSM_STREAM_DEFINE(64, 8, 4)
SSM_STREAM_DEFINE(64, 16, 2)
}  // namespace stream
}  // namespace ssm
