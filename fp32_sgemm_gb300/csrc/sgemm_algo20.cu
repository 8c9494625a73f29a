// Main-kernel instantiation for tile configuration 20: 256 x 128 output
// tile, eight consumer warps in one CTA per SM, 16-deep K slices and 6
// stages, 8-byte A and 16-byte B fragments both double buffered, C read and
// written from registers.  For short K that is not a multiple of 32 (16, 48,
// ...) with beta != 0 and an aligned C, where 32-deep slices would multiply
// zero padding.
#include "kernel_table.h"

namespace sg {
using CfgAlgo20 = FfmaConfig<256,128,16,6,4,2,8,4,1,2,1>;
void fill_algo20(KernelEntry *v) { fill_variants<CfgAlgo20>(v); }
}  // namespace sg
