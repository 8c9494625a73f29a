// Main-kernel instantiation for tile configuration 24: 256 x 128 output
// tile, eight consumer warps in one CTA per SM, 8-deep K slices and 8
// stages, 16-byte A reads double buffered one k ahead, C through per-warp
// shared-memory staging.  For short K that is not a multiple of 16.
#include "kernel_table.h"

namespace sg {
using CfgAlgo24 = FfmaConfig<256,128,8,8,4,2,8,2,1,4,0,1>;
void fill_algo24(KernelEntry *v) { fill_variants<CfgAlgo24>(v); }
}  // namespace sg
