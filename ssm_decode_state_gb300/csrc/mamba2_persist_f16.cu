// The persistent Mamba-2 replay decode for an FP16 checkpoint (stochastic
// rounding at flushes); a translation unit of its own so that it compiles in
// parallel with the float32 instantiations.
#include "mamba2_persist_launch.cuh"

namespace rssm {

rssm_status launch_decode_persistent_f16(const rssm_mamba2_dims *d, const M2Args &args, cudaStream_t st) {
    return launch_decode_persistent_ck<1>(d, args, st);
}

}  // namespace rssm
