// FP16, K-major B: the single-CTA kernels of this operand kind and layout.
#include "launch.h"
namespace dgt {
DGT_DEFINE_VARIANTS(f16_km, KIND_F16, true)
}  // namespace dgt
