// STREAM instances for 32 states (kernel template in stream_core.cuh).
#include "stream_core.cuh"

namespace ssm {
namespace stream {
SSM_STREAM_DEFINE(32, 4, 4)
SSM_STREAM_DEFINE(32, 8, 2)
SSM_STREAM_DEFINE(32, 8, 4)
}  // namespace stream
}  // namespace ssm
