// thc_p16.cu -- the fused THC kernels built for exactly 16 workers (see thc_fused.cuh).
#include "thc_fused.cuh"

namespace gar {
namespace thc {
template int launch_fused<16>(const FusedParams &, int, bool, cudaStream_t);
template int launch_fused_plan<16>(const ThcPlanParams &, int, bool, bool, cudaStream_t);
}  // namespace thc
}  // namespace gar
