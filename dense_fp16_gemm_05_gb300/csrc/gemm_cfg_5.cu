// gemm_cfg_5.cu -- kernel instances of configuration 5 (2sm_256x512_s4): ReLU on and
// off, all four operand layouts (NN, NT, TN, TT).  One translation unit per configuration so that
// the instances compile in parallel.
#include "gemm_launch.cuh"

namespace gemm_sm103 {

int launch_config_5(const LaunchArgs &a) { return launch_config<Cfg2x512, true>(a); }

int launch_info_config_5(int64_t M, int64_t N, bool allow_split, const DeviceInfo &dev, int *grid_ctas,
                         int *cluster_size, int *tiles)
{
    return config_launch_info<Cfg2x512>(M, N, allow_split, dev, grid_ctas, cluster_size, tiles);
}

double wave_eff_config_5(int64_t M, int64_t N, bool allow_split, const DeviceInfo &dev)
{
    return config_wave_efficiency<Cfg2x512>(M, N, allow_split, dev);
}

}  // namespace gemm_sm103
