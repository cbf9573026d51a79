// BF16, row-major B: the CTA-pair kernels of this operand kind and layout.
#include "launch.h"
namespace dgt {
DGT_DEFINE_PAIR_VARIANTS(bf16_rm, KIND_BF16, false)
}  // namespace dgt
