// gemm_cfg_6.cu -- kernel instances of configuration 6 (4sm_512x256_mc_s6): ReLU on and
// off, the NN layout only.  One translation unit per configuration so that
// the instances compile in parallel.
#include "gemm_launch.cuh"

namespace gemm_sm103 {

int launch_config_6(const LaunchArgs &a) { return launch_config<Cfg4x256mc, false>(a); }

int launch_info_config_6(int64_t M, int64_t N, bool allow_split, const DeviceInfo &dev, int *grid_ctas,
                         int *cluster_size, int *tiles)
{
    return config_launch_info<Cfg4x256mc>(M, N, allow_split, dev, grid_ctas, cluster_size, tiles);
}

double wave_eff_config_6(int64_t M, int64_t N, bool allow_split, const DeviceInfo &dev)
{
    return config_wave_efficiency<Cfg4x256mc>(M, N, allow_split, dev);
}

}  // namespace gemm_sm103
