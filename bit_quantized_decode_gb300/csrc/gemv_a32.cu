// Weight-only GEMVs on float activations (formats W4F and W8F, xmode X_F32):
// the paths "Jetson Orin AGX INT4 推理优化实践" §"为什么 INT4 float 解包不快"
// measures INT4 DP4A against, built on the same streaming kernel so that only
// the inner loop differs.  One to four tokens.
#include "gemv_kernel.cuh"

namespace w4k {

namespace {

template <int FMT>
cudaError_t launch_a32_fmt(const ChainParams<1>& p, int MT, int grid, size_t smem, bool pdl, cudaStream_t s)
{
    switch (MT) {
        case 1: return launch_gemv_t<FMT, 1, X_F32>(p, grid, smem, pdl, s);
        case 2: return launch_gemv_t<FMT, 2, X_F32>(p, grid, smem, pdl, s);
        case 4: return launch_gemv_t<FMT, 4, X_F32>(p, grid, smem, pdl, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_gemv_a32(int fmt, const ChainParams<1>& p, int MT, int grid, size_t smem, bool pdl,
                            cudaStream_t s)
{
    if (fmt == FMT_W4F) return launch_a32_fmt<FMT_W4F>(p, MT, grid, smem, pdl, s);
    if (fmt == FMT_W8F) return launch_a32_fmt<FMT_W8F>(p, MT, grid, smem, pdl, s);
    return cudaErrorInvalidValue;
}

}  // namespace w4k
