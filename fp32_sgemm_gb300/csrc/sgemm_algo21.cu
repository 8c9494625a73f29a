// Main-kernel instantiation for tile configuration 21: configuration 15
// (256 x 128, eight warps, one CTA per SM) with 8-deep K slices and 8
// stages.  For K of 8 or 24 and the like.
#include "kernel_table.h"

namespace sg {
using CfgAlgo21 = FfmaConfig<256,128,8,8,4,2,8,4,1,2,0,1>;
void fill_algo21(KernelEntry *v) { fill_variants<CfgAlgo21>(v); }
}  // namespace sg
