// Main-kernel instantiation for tile configuration 23: 256 x 128 output
// tile, eight consumer warps in one CTA per SM, 16-deep K slices and 4
// stages, 16-byte A reads double buffered one k ahead, C through per-warp
// shared-memory staging (TMA tile stores when beta == 0 and C is aligned,
// row runs when C is not aligned).  For short K that is a multiple of 16 but
// not of 32.
#include "kernel_table.h"

namespace sg {
using CfgAlgo23 = FfmaConfig<256,128,16,4,4,2,8,4,1,4,0,1>;
void fill_algo23(KernelEntry *v) { fill_variants<CfgAlgo23>(v); }
}  // namespace sg
