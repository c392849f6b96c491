// bf16 instantiations of the split-KV and combine kernels.
#include "splitkv_launch.cuh"

namespace pa {
int launch_splitkv_bf16(const Args& a, const SplitPlan& plan, void* workspace, unsigned int* err, char* msg,
                        size_t msg_len) {
    return launch_splitkv_t<__nv_bfloat16>(a, plan, workspace, err, msg, msg_len);
}
int splitkv_occupancy_bf16(const SplitPlan& plan) { return splitkv_occupancy_t<__nv_bfloat16>(plan); }
}  // namespace pa
