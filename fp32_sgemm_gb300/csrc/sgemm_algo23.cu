// Main-kernel instantiation for tile configuration 23: configuration 20
// (256 x 128, 16-deep K slices) with 4 stages, C stored by TMA from
// per-warp shared-memory staging, and the 16-byte A loop of configuration 28.
#include "kernel_table.h"

namespace sg {
using CfgAlgo23 = FfmaConfig<256,128,16,4,4,2,8,4,1,4,0,2,0,1>;
void fill_algo23(KernelEntry *v) { fill_variants<CfgAlgo23>(v); }
}  // namespace sg
