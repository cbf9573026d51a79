// BF16 instantiations of the GEMM kernel.
#include "launch.h"
namespace dgt {
cudaError_t launch_bf16(const LaunchPlan& L) { return launch_kind<KIND_BF16>(L); }
}  // namespace dgt
