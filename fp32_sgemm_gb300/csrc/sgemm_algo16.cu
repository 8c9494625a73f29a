// Main-kernel instantiation for tile configuration 16: 64 x 512 output tile,
// eight consumer warps (1 x 8 warp tiles of 64 x 64) in one CTA per SM,
// BK=32, 3 stages (B in two 256-column TMA boxes), 16-byte A reads double
// buffered one k ahead, each k's B read just before its FMAs.  For products
// with 33 to 64 rows.
#include "kernel_table.h"

namespace sg {
using CfgAlgo16 = FfmaConfig<64,512,32,3,1,8,8,4,1,4,0>;
void fill_algo16(KernelEntry *v) { fill_variants<CfgAlgo16>(v); }
}  // namespace sg
