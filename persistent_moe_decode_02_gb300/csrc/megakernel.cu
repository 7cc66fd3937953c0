// Host entry points of the megakernel: the launches, the RoPE table and the
// shared-memory bookkeeping.  The device code is in megakernel.cuh; the
// kernel instances with the nucleus-draw tasks are built in megakernel_nuc.cu,
// so the greedy and temperature kernels carry none of that code.
#include "megakernel.cuh"

namespace mk {
cudaError_t launch_megakernel_nuc(const Params& p, int nb, int grid, int smem, cudaStream_t st);
int max_active_ctas_nuc(int nb, int smem);
namespace {

__global__ void k_rope_table(float2* tab, int npos, int half, int d, double theta) {
  const long long n = (long long)npos * half;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int pos = (int)(idx / half), i = (int)(idx % half);
    const double inv = pow(theta, -2.0 * i / d);
    double s, c;
    sincos((double)pos * inv, &s, &c);
    tab[idx] = make_float2((float)c, (float)s);
  }
}

}  // namespace

// The nucleus-draw instance runs only when the LM tiles keep their logits
// for the draw tasks; every other step takes the plain instance.
cudaError_t launch_megakernel(const Params& p, int nb, int grid, int smem, cudaStream_t st) {
  if (p.lg_keep) return launch_megakernel_nuc(p, nb, grid, smem, st);
  switch (nb) {
    case 1: return launch_nb<1, false>(p, grid, smem, st);
    case 2: return launch_nb<2, false>(p, grid, smem, st);
    case 4: return launch_nb<4, false>(p, grid, smem, st);
    case 8: return launch_nb<8, false>(p, grid, smem, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_rope_table(float2* tab, int npos, int d, double theta, cudaStream_t st) {
  const int half = d / 2;
  long long n = (long long)npos * half;
  int blocks = (int)((n + 255) / 256);
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  k_rope_table<<<blocks, 256, 0, st>>>(tab, npos, half, d, theta);
  return cudaGetLastError();
}

// Resident CTAs per SM of both instances (the smaller of the two).
int max_active_ctas(int nb, int smem) {
  int n = 0;
  switch (nb) {
    case 1: n = occupancy<1, false>(smem); break;
    case 2: n = occupancy<2, false>(smem); break;
    case 4: n = occupancy<4, false>(smem); break;
    case 8: n = occupancy<8, false>(smem); break;
    default: return 0;
  }
  const int m = max_active_ctas_nuc(nb, smem);
  return n < m ? n : m;
}

size_t misc_bytes() { return sizeof(Misc); }

}  // namespace mk
