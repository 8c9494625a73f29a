// Main-kernel instantiation for tile configuration 28: configuration 22
// with 16-byte A reads, only the A fragments double buffered, and four A
// groups per unrolled loop iteration.
#include "kernel_table.h"

namespace sg {
using CfgAlgo28 = FfmaConfig<256,128,32,2,4,2,8,4,1,4,0,2,0,1,0>;
void fill_algo28(KernelEntry *v) { fill_variants<CfgAlgo28>(v); }
}  // namespace sg
