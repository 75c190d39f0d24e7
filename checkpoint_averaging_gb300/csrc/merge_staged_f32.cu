// merge_staged_f32.cu -- the staged merge pass for fp32 worker checkpoints.
#include "merge_staged.cuh"

namespace cam {

MergeFn pick_staged_f32(const MergeVariant& v) { return dev::staged_for_dtype<float>(v); }

}  // namespace cam
