// STREAM instances for 4 and 8 states (kernel template in stream_core.cuh).
#include "stream_core.cuh"

namespace ssm {
namespace stream {
SSM_STREAM_DEFINE(4, 4, 2)
SSM_STREAM_DEFINE(4, 4, 4)
SSM_STREAM_DEFINE(8, 4, 2)
SSM_STREAM_DEFINE(8, 4, 4)
SSM_STREAM_DEFINE(8, 8, 2)
}  // namespace stream
}  // namespace ssm
