// Main-kernel instantiation for tile configuration 17: 512 x 64 output tile,
// eight consumer warps (8 x 1 warp tiles of 64 x 64) in one CTA per SM,
// BK=32, 3 stages (A in two 256-row TMA boxes), 16-byte A reads double
// buffered one k ahead, each k's B read just before its FMAs.  For products
// with 33 to 64 columns.
#include "kernel_table.h"

namespace sg {
using CfgAlgo17 = FfmaConfig<512,64,32,3,8,1,8,4,1,4,0>;
void fill_algo17(KernelEntry *v) { fill_variants<CfgAlgo17>(v); }
}  // namespace sg
