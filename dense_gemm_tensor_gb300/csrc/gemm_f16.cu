// FP16 instantiations of the GEMM kernel.
#include "launch.h"
namespace dgt {
cudaError_t launch_f16(const LaunchPlan& L) { return launch_kind<KIND_F16>(L); }
int pair_clusters_f16(bool kmajor, int bn, int pairs) { return pair_clusters_kind<KIND_F16>(kmajor, bn, pairs); }
}  // namespace dgt
