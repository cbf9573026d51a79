// BF16, K-major B: the CTA-pair kernels of this operand kind and layout.
#include "launch.h"
namespace dgt {
DGT_DEFINE_PAIR_VARIANTS(bf16_km, KIND_BF16, true)
}  // namespace dgt
