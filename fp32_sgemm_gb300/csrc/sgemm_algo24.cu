// Main-kernel instantiation for tile configuration 24: configuration 21
// (256 x 128, 8-deep K slices, 8 stages) with C stored by TMA from
// per-warp shared-memory staging and the 16-byte A loop of configuration 28.
#include "kernel_table.h"

namespace sg {
using CfgAlgo24 = FfmaConfig<256,128,8,8,4,2,8,2,1,4,0,2,0,1>;
void fill_algo24(KernelEntry *v) { fill_variants<CfgAlgo24>(v); }
}  // namespace sg
