// GEMV kernels for one weight format, kept in a translation unit of their own
// so the formats compile in parallel.
#include "gemv_kernel.cuh"

namespace w4k {

cudaError_t launch_gemv_w4(const ChainParams<1>& p, int MT, int xmode, int grid, size_t smem, bool pdl,
                          cudaStream_t s)
{
    return launch_gemv_fmt<FMT_W4>(p, MT, xmode, grid, smem, pdl, s);
}

}  // namespace w4k
