// BF16, K-major B: the single-CTA kernels of this operand kind and layout.
#include "launch.h"
namespace dgt {
DGT_DEFINE_VARIANTS(bf16_km, KIND_BF16, true)
}  // namespace dgt
