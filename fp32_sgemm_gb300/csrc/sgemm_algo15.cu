// Main-kernel instantiation for tile configuration 15: 256 x 128 output
// tile, eight consumer warps (4 x 2 warp tiles of 64 x 64) in one CTA per SM,
// BK=32, 4 stages, TMA issued by thread 0, double-buffered fragments.
#include "kernel_table.h"

namespace sg {
using CfgAlgo15 = FfmaConfig<256,128,32,4,4,2,8,4,1,2,0,1>;
void fill_algo15(KernelEntry *v) { fill_variants<CfgAlgo15>(v); }
}  // namespace sg
