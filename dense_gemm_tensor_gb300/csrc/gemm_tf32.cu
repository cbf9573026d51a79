// TF32 instantiations of the GEMM kernel.
#include "launch.h"
namespace dgt {
cudaError_t launch_tf32(const LaunchPlan& L) { return launch_kind<KIND_TF32>(L); }
int pair_clusters_tf32(bool kmajor, int bn, int pairs) { return pair_clusters_kind<KIND_TF32>(kmajor, bn, pairs); }
}  // namespace dgt
