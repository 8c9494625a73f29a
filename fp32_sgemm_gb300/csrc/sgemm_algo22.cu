// Main-kernel instantiation for tile configuration 22: configuration 15
// (256 x 128, eight warps, one CTA per SM, 32-deep K slices) with 2 stages,
// refilled as soon as every warp released a slice, and C stored through
// per-warp shared-memory staging and TMA tile stores, so that writing C
// overlaps the next tile's arithmetic (short K).
#include "kernel_table.h"

namespace sg {
using CfgAlgo22 = FfmaConfig<256,128,32,2,4,2,8,4,1,2,0,1,0,1,0>;
void fill_algo22(KernelEntry *v) { fill_variants<CfgAlgo22>(v); }
}  // namespace sg
