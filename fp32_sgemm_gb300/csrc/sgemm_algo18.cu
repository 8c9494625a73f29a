// Main-kernel instantiation for tile configuration 18: 32 x 1024 output
// tile, eight consumer warps (1 x 8 warp tiles of 32 x 128, lane grid 4 x 8)
// in one CTA per SM, BK=16, 3 stages (B in four 256-column TMA boxes),
// 8-byte A and 16-byte B fragments both double buffered.  For large products
// with 17 to 32 rows.
#include "kernel_table.h"

namespace sg {
using CfgAlgo18 = FfmaConfig<32,1024,16,3,1,8,4,4,1,2,1>;
void fill_algo18(KernelEntry *v) { fill_variants<CfgAlgo18>(v); }
}  // namespace sg
