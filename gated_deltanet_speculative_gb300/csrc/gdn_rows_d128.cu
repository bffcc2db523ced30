// gdn_rows_d128.cu -- row kernels (step, window, tree) for d_k = d_v = 128.
#include "gdn_launch.h"

namespace gdn {
cudaError_t launch_rows_d128(int mode, const RowParams &p, int n_streams, cudaStream_t st) {
    return launch_rows<128>(mode, p, n_streams, st);
}
}  // namespace gdn
