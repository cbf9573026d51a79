// TF32, row-major B: the CTA-pair kernels of this operand kind and layout.
#include "launch.h"
namespace dgt {
DGT_DEFINE_PAIR_VARIANTS(tf32_rm, KIND_TF32, false)
}  // namespace dgt
