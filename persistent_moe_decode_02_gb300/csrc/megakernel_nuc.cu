// The megakernel instances with nucleus (top-p) draw tasks compiled in.  They
// are built in a translation unit of their own, in parallel with the plain
// instances of megakernel.cu, whose code therefore holds none of the draw.
#include "megakernel.cuh"

namespace mk {

cudaError_t launch_megakernel_nuc(const Params& p, int nb, int grid, int smem, cudaStream_t st) {
  switch (nb) {
    case 1: return launch_nb<1, true>(p, grid, smem, st);
    case 2: return launch_nb<2, true>(p, grid, smem, st);
    case 4: return launch_nb<4, true>(p, grid, smem, st);
    case 8: return launch_nb<8, true>(p, grid, smem, st);
    default: return cudaErrorInvalidValue;
  }
}

int max_active_ctas_nuc(int nb, int smem) {
  switch (nb) {
    case 1: return occupancy<1, true>(smem);
    case 2: return occupancy<2, true>(smem);
    case 4: return occupancy<4, true>(smem);
    case 8: return occupancy<8, true>(smem);
    default: return 0;
  }
}

}  // namespace mk
