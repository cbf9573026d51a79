// FP16, row-major B: the CTA-pair kernels of this operand kind and layout.
#include "launch.h"
namespace dgt {
DGT_DEFINE_PAIR_VARIANTS(f16_rm, KIND_F16, false)
}  // namespace dgt
