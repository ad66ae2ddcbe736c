// NVFP4 top-k with the hidden width unrolled at compile time (K = 2,560 and
// 5,120, up to 4 hidden rows per launch).
#include "argmax_lowbit.cuh"

namespace dvl {
namespace lowbit {

template cudaError_t launch_kc<kFmtNvfp4, 4>(const ArgmaxArgs &, int, cudaStream_t);

}  // namespace lowbit
}  // namespace dvl
