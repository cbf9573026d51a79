// FP16, row-major B: the single-CTA kernels of this operand kind and layout.
#include "launch.h"
namespace dgt {
DGT_DEFINE_VARIANTS(f16_rm, KIND_F16, false)
}  // namespace dgt
