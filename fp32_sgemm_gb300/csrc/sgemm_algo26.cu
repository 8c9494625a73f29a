// Main-kernel instantiation for tile configuration 26: configuration 14
// (128 x 256, eight warps, one CTA per SM, 32-deep K slices) with 2 stages,
// refilled as soon as every warp released a slice, and C stored by TMA
// from per-warp shared-memory staging.
#include "kernel_table.h"

namespace sg {
using CfgAlgo26 = FfmaConfig<128,256,32,2,2,4,8,4,1,2,0,1,0,1,0>;
void fill_algo26(KernelEntry *v) { fill_variants<CfgAlgo26>(v); }
}  // namespace sg
