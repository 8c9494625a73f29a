// Main-kernel instantiation for tile configuration 10: 128 x 128 output
// tile, four consumer warps (2 x 2 warp tiles of 64 x 64), two CTAs per SM,
// BK=32, 3 stages, 8-byte A and 16-byte B fragments both double buffered.
// For matrices of at most 128 x 128 that reach the tile kernel (large
// batches of small products): the tile that wastes the fewest lanes.
#include "kernel_table.h"

namespace sg {
using CfgAlgo10 = FfmaConfig<128,128,32,3,2,2,8,4,2,2,1>;
void fill_algo10(KernelEntry *v) { fill_variants<CfgAlgo10>(v); }
}  // namespace sg
