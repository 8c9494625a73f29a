// Main-kernel instantiation for tile configuration 13: 256 x 64 output
// tile (one warp column of four 64 x 64 warp tiles), BK=32, 2 stages, TMA
// issued by thread 0, double-buffered fragments, 2 CTAs/SM.  For products
// with at most 64 columns.
#include "kernel_table.h"

namespace sg {
using CfgAlgo13 = FfmaConfig<256,64,32,2,4,1,8,4,2,2,0,1>;
void fill_algo13(KernelEntry *v) { fill_variants<CfgAlgo13>(v); }
}  // namespace sg
