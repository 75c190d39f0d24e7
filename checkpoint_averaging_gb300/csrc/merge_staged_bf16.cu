// merge_staged_bf16.cu -- the staged merge pass for bf16 worker checkpoints
// (widened to fp32 on the way out of shared memory; the widening is exact).
#include "merge_staged.cuh"

namespace cam {

MergeFn pick_staged_bf16(const MergeVariant& v) { return dev::staged_for_dtype<uint16_t>(v); }

}  // namespace cam
