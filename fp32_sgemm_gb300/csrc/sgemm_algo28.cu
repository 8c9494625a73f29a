// Main-kernel instantiation for tile configuration 28: 256 x 128 output
// tile, eight consumer warps (4 x 2 warp tiles of 64 x 64) in one CTA per
// SM, BK=32, a 2-stage ring refilled as soon as every warp released a slice,
// 16-byte A reads double buffered one k ahead (four A groups per unrolled
// iteration), each k's B read just before its FMAs, C through per-warp
// shared-memory staging: TMA tile stores when beta == 0 and C is aligned
// (the automatic choice from 256 rows up), row runs of plain stores when C
// is not aligned.
#include "kernel_table.h"

namespace sg {
using CfgAlgo28 = FfmaConfig<256,128,32,2,4,2,8,4,1,4,0,1,0>;
void fill_algo28(KernelEntry *v) { fill_variants<CfgAlgo28>(v); }
}  // namespace sg
