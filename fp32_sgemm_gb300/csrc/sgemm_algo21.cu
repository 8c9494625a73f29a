// Main-kernel instantiation for tile configuration 21: 256 x 128 output
// tile, eight consumer warps in one CTA per SM, 8-deep K slices and 8
// stages, both fragments double buffered, C from registers.  For K of 8, 24
// and the like with beta != 0 and an aligned C.
#include "kernel_table.h"

namespace sg {
using CfgAlgo21 = FfmaConfig<256,128,8,8,4,2,8,4,1,2,1>;
void fill_algo21(KernelEntry *v) { fill_variants<CfgAlgo21>(v); }
}  // namespace sg
