// Main-kernel instantiation for tile configuration 25: configuration 23
// (256 x 128, 16-deep K slices, 4 stages, C stored by TMA) with each stage
// refilled as soon as every warp released it.
#include "kernel_table.h"

namespace sg {
using CfgAlgo25 = FfmaConfig<256,128,16,4,4,2,8,4,1,2,0,1,0,1,0>;
void fill_algo25(KernelEntry *v) { fill_variants<CfgAlgo25>(v); }
}  // namespace sg
