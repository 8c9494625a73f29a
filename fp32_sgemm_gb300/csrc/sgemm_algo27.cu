// Main-kernel instantiation for tile configuration 27: 128 x 256 output
// tile, eight consumer warps (2 x 4 warp tiles of 64 x 64) in one CTA per
// SM, BK=32, a 2-stage ring refilled as soon as every warp released a slice,
// 16-byte A reads double buffered one k ahead, each k's B read just before
// its FMAs, C through per-warp shared-memory staging.  The wide-product form
// of configuration 28.
#include "kernel_table.h"

namespace sg {
using CfgAlgo27 = FfmaConfig<128,256,32,2,2,4,8,4,1,4,0,1,0>;
void fill_algo27(KernelEntry *v) { fill_variants<CfgAlgo27>(v); }
}  // namespace sg
