// merge_fused_f32.cu -- the fused merge pass for fp32 worker checkpoints.
#include "merge_fused.cuh"

namespace cam {

MergeFn pick_merge_f32(const MergeVariant& v) { return dev::pick_for_dtype<float>(v); }

}  // namespace cam
