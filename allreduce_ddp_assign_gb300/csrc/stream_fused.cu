// The streaming kernel's fused pack + ring-reduce (+ copy-back) instantiations.
#include "stream_impl.cuh"

namespace ddpk {
ddp_status launch_stream_fused(StreamArgs& a, int dtype, void* stream) { return launch_op<OP_FUSED>(a, dtype, stream); }
}  // namespace ddpk
