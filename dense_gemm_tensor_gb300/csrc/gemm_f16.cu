// FP16 instantiations of the GEMM kernel.
#include "launch.h"
namespace dgt {
cudaError_t launch_f16(const LaunchPlan& L) { return launch_kind<KIND_F16>(L); }
}  // namespace dgt
