// STREAM instances for 16 states (kernel template in stream_core.cuh).
#include "stream_core.cuh"

namespace ssm {
namespace stream {
SSM_STREAM_DEFINE(16, 4, 4)
SSM_STREAM_DEFINE(16, 8, 2)
SSM_STREAM_DEFINE(16, 8, 4)
SSM_STREAM_DEFINE(16, 16, 2)
}  // namespace stream
}  // namespace ssm
