// merge_fused_bf16.cu -- the fused merge pass for bf16 worker checkpoints
// (widened to fp32 in registers; the widening is exact).
#include "merge_fused.cuh"

namespace cam {

MergeFn pick_merge_bf16(const MergeVariant& v) { return dev::pick_for_dtype<uint16_t>(v); }

}  // namespace cam
