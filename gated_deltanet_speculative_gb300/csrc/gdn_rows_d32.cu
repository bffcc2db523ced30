// gdn_rows_d32.cu -- row kernels (step, window, tree) for d_k = d_v = 32.
#include "gdn_launch.h"

namespace gdn {
cudaError_t launch_rows_d32(int mode, const RowParams &p, int n_streams, cudaStream_t st) {
    return launch_rows<32>(mode, p, n_streams, st);
}
}  // namespace gdn
