// FP16, row-major B: every GEMM kernel instantiation of this operand kind and layout.
#include "launch.h"
namespace dgt {
DGT_DEFINE_VARIANTS(f16_rm, KIND_F16, false)
}  // namespace dgt
