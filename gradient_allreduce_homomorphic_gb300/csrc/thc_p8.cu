// thc_p8.cu -- the fused THC kernels built for exactly 8 workers (see thc_fused.cuh).
#include "thc_fused.cuh"

namespace gar {
namespace thc {
template int launch_fused<8>(const FusedParams &, int, bool, cudaStream_t);
template int launch_fused_plan<8>(const ThcPlanParams &, int, bool, bool, cudaStream_t);
}  // namespace thc
}  // namespace gar
