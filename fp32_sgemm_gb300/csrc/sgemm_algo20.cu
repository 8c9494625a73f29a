// Main-kernel instantiation for tile configuration 20: configuration 15
// (256 x 128, eight warps, one CTA per SM) with 16-deep K slices and 6
// stages.  For short K (16, 48, ...), where 32-deep slices would multiply
// zero padding; there the product is bound by writing C.
#include "kernel_table.h"

namespace sg {
using CfgAlgo20 = FfmaConfig<256,128,16,6,4,2,8,4,1,2,0,1>;
void fill_algo20(KernelEntry *v) { fill_variants<CfgAlgo20>(v); }
}  // namespace sg
