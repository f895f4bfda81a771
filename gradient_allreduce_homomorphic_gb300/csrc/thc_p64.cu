// thc_p64.cu -- the fused THC kernels built for exactly 64 workers (see thc_fused.cuh).
#include "thc_fused.cuh"

namespace gar {
namespace thc {
template int launch_fused<64>(const FusedParams &, int, bool, cudaStream_t);
template int launch_fused_plan<64>(const ThcPlanParams &, int, bool, bool, cudaStream_t);
}  // namespace thc
}  // namespace gar
