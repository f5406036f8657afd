// sm_103a tensor-core path (tcgen05 / TMEM / TMA).  Placeholder until the
// kernels land: reports every shape as unsupported so the SIMT path runs.
#include "tri_attn_internal.h"

namespace tri_attn {

bool sm103_supported(int, int, int, int) { return false; }
Workspace sm103_layout(int I, int) { Workspace w; w.I = I; w.I_pad = round_up(I, kTile); return w; }
cudaError_t sm103_forward(const FwdArgs&, cudaStream_t, LaunchTimer*) { return cudaErrorNotSupported; }

}  // namespace tri_attn
