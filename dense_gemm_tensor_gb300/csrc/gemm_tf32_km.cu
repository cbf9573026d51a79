// TF32, K-major B: the single-CTA kernels of this operand kind and layout.
#include "launch.h"
namespace dgt {
DGT_DEFINE_VARIANTS(tf32_km, KIND_TF32, true)
}  // namespace dgt
