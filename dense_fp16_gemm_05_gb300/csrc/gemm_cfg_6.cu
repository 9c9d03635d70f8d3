// gemm_cfg_6.cu -- kernel instances of configuration 6 (1sm_128x128_ck_s6): single-CTA
// 128 x 128 tiles whose K loop is split over a cluster of 1, 2, 4 or 8 CTAs, the
// partial tiles added through distributed shared memory; ReLU on and off, NN layout.
// One translation unit per configuration so that the instances compile in parallel.
#include "gemm_launch.cuh"

namespace gemm_sm103 {

int launch_config_6(const LaunchArgs &a)
{
    if (a.transa || a.transb) return GEMM_ERR_INVALID_ARG;
    return a.relu ? launch_one_ck<Cfg1x128ck, true>(a) : launch_one_ck<Cfg1x128ck, false>(a);
}

// Without a K: the geometry of clusters of one CTA.
int launch_info_config_6(int64_t M, int64_t N, bool, const DeviceInfo &dev, int *grid_ctas, int *cluster_size,
                         int *tiles)
{
    return ck_launch_info<Cfg1x128ck>(M, N, 64, 1, dev, grid_ctas, cluster_size, tiles);
}

double wave_eff_config_6(int64_t M, int64_t N, bool, const DeviceInfo &dev)
{
    return ck_wave_efficiency<Cfg1x128ck>(M, N, 64, 1, dev);
}

int ck_launch_info_config_6(int64_t M, int64_t N, int64_t K, int request, const DeviceInfo &dev, int *grid_ctas,
                            int *cluster_size, int *tiles)
{
    return ck_launch_info<Cfg1x128ck>(M, N, K, request, dev, grid_ctas, cluster_size, tiles);
}

double ck_wave_eff_config_6(int64_t M, int64_t N, int64_t K, int request, const DeviceInfo &dev)
{
    return ck_wave_efficiency<Cfg1x128ck>(M, N, K, request, dev);
}

}  // namespace gemm_sm103
