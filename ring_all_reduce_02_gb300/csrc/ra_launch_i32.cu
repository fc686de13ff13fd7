// Kernel instantiations for one dtype (compiled as its own translation unit so
// the four dtypes build in parallel).
#include "ra_kernels.cuh"
#include "ra_order.cuh"

namespace ra {
cudaError_t launch_i32(int kind, int op, const Args& a, dim3 grid, cudaStream_t s) {
  return launch_dtype<DT_I32>(kind, op, a, grid, s);
}
cudaError_t launch_ordered_i32(bool is_rs, int op, const OrderArgs& o, dim3 grid, cudaStream_t s) {
  return launch_ordered_dtype<DT_I32>(is_rs, op, o, grid, s);
}
}  // namespace ra
