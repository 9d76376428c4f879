// Split kernel dispatch (transitional: the scalar kernel until the tensor-core kernel lands).
#include "smla_internal.h"

namespace smla {

bool split_shape_supported(int H, int topk) {
  return (H == 16 || H == 32 || H == 64 || H == 128) && topk >= 1 && topk <= kMaxTopk;
}

int split_ctas_per_sm(int H) { (void)H; return 1; }

cudaError_t launch_split_tc(const SplitParams& p, cudaStream_t stream) { return launch_split_simt(p, stream); }

}  // namespace smla
