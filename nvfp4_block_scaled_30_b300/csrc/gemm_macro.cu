// Placeholder for the FP16 macro-scale contraction (see launch_w4a4_macro).
#include "internal.h"

namespace nv4 {

cudaError_t launch_w4a4_macro(const MacroGemmArgs &, cudaStream_t) { return cudaErrorNotSupported; }

} // namespace nv4
