// TF32, row-major B: the CTA-pair kernel on the transposed product C^T = B^T A^T, each tile width.
#include "launch.h"
namespace dgt {
DGT_DEFINE_SWAP_VARIANTS(tf32_sw, KIND_TF32)
}  // namespace dgt
