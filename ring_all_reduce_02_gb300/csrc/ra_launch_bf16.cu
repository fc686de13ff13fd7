// Kernel instantiations for one dtype (compiled as its own translation unit so
// the four dtypes build in parallel).
#include "ra_kernels.cuh"
#include "ra_order.cuh"

namespace ra {
cudaError_t launch_bf16(int kind, int op, const Args& a, dim3 grid, cudaStream_t s) {
  return launch_dtype<DT_BF16>(kind, op, a, grid, s);
}
cudaError_t launch_ordered_bf16(bool is_rs, int op, const OrderArgs& o, dim3 grid, cudaStream_t s) {
  return launch_ordered_dtype<DT_BF16>(is_rs, op, o, grid, s);
}
}  // namespace ra
