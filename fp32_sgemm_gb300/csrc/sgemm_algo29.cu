// Main-kernel instantiation for tile configuration 29: 256 x 128 output
// tile, eight consumer warps in one CTA per SM, BK=32, 4 stages refilled one
// slice late, the inner loop of configuration 28, C read and written from
// registers with 16-byte accesses.  The automatic choice when beta != 0 and
// C is 16-byte aligned.
#include "kernel_table.h"

namespace sg {
using CfgAlgo29 = FfmaConfig<256,128,32,4,4,2,8,4,1,4,0>;
void fill_algo29(KernelEntry *v) { fill_variants<CfgAlgo29>(v); }
}  // namespace sg
