// gemm_cfg_1.cu -- kernel instances of configuration 1 (1sm_128x256_s4): ReLU on and
// off, all four operand layouts (NN, NT, TN, TT).  One translation unit per configuration so that
// the instances compile in parallel.
#include "gemm_launch.cuh"

namespace gemm_sm103 {

int launch_config_1(const LaunchArgs &a) { return launch_config<Cfg1x256, true>(a); }

int launch_info_config_1(int64_t M, int64_t N, bool allow_split, const DeviceInfo &dev, int *grid_ctas,
                         int *cluster_size, int *tiles)
{
    return config_launch_info<Cfg1x256>(M, N, allow_split, dev, grid_ctas, cluster_size, tiles);
}

double wave_eff_config_1(int64_t M, int64_t N, bool allow_split, const DeviceInfo &dev)
{
    return config_wave_efficiency<Cfg1x256>(M, N, allow_split, dev);
}

}  // namespace gemm_sm103
