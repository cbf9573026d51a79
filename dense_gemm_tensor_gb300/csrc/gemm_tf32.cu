// TF32 instantiations of the GEMM kernel.
#include "launch.h"
namespace dgt {
cudaError_t launch_tf32(const LaunchPlan& L) { return launch_kind<KIND_TF32>(L); }
}  // namespace dgt
