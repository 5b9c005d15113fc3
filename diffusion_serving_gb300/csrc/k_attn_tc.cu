// Tensor-core chunk attention (placeholder until the tcgen05 kernel lands).
#include "kvc_internal.h"

bool kvc_tc_supported(const kvc_config&) { return false; }
bool kvc_tc_make_kv_maps(kvc_cache*) { return false; }
cudaError_t kvc_launch_attn_tc(kvc_cache*, const void*, void*, int, bool, cudaStream_t) {
  return cudaErrorNotSupported;
}
