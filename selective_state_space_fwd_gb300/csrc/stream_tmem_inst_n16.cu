// STREAM-TM instances for 16 states: 4 states per lane; one channel per lane
// (8 compute warps per CTA) or a channel pair (4 compute warps).
#include "stream_tmem_launch.cuh"

namespace ssm {
namespace stream_tm {
SSM_TM_DEFINE(16, 4, 1, 8)
SSM_TM_DEFINE(16, 4, 2, 4)
}  // namespace stream_tm
}  // namespace ssm
