// Main-kernel instantiation for tile configuration 19: 1024 x 32 output
// tile, eight consumer warps (8 x 1 warp tiles of 128 x 32, lane grid 16 x
// 2) in one CTA per SM, BK=16, 3 stages (A in four 256-row TMA boxes),
// 8-byte A and 16-byte B fragments both double buffered.  For large products
// with 17 to 32 columns.
#include "kernel_table.h"

namespace sg {
using CfgAlgo19 = FfmaConfig<1024,32,16,3,8,1,16,4,1,2,1>;
void fill_algo19(KernelEntry *v) { fill_variants<CfgAlgo19>(v); }
}  // namespace sg
